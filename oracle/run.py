"""The oracle on a seeded workload: draws the same inputs on the host and runs the fp64
oracle one sequence at a time.

TEST INFRASTRUCTURE ONLY (tests, the smoke check and the benchmark's CPU baseline).
Inputs come from the shared counter-based generator (torch CPU, converted to numpy);
every computation of the method is the numpy code of dflash_oracle.
"""
from __future__ import annotations

import numpy as np

from workload import inputs
from workload.configs import Workload

from . import dflash_oracle as O


def np64(t):
    return t.float().numpy().astype(np.float64) if t.dtype != np.float64 else t


def host_weights(w: Workload):
    """All drafter weights as fp32 numpy arrays (exact copies of the bf16/fp32 values;
    numpy promotes them to fp64 inside every product).  For FP8 workloads the projection
    matrices are the oracle's own dequantized FP8 form of those values."""
    W = {n: inputs.weight(w, n, s, k).float().numpy() for n, s, k in inputs.weight_specs(w)}
    return O.fp8_weights(W) if w.weight_format == "fp8" else W


def context(w: Workload, W, b, p0, p1):
    """Fused features and per-layer injected K/V of sequence b, positions [p0, p1)."""
    bf16 = w.dtype == "bf16"
    x = np64(inputs.ctx_hidden(w, b, p0, p1))
    fused = O.fuse_features(x, W["w_fuse"], W["g_fuse"], w.rms_eps, bf16)
    K, V = [], []
    pos = np.arange(p0, p1)
    for l in range(w.n_layers):
        k, v = O.inject_kv(fused, pos, W[f"l{l}.w_k"], W[f"l{l}.w_v"], w.n_kv_heads,
                           w.rope_theta, bf16)
        K.append(k)
        V.append(v)
    return fused, K, V


def draft_sequence(w: Workload, W, b, ctx=None):
    """Oracle draft of sequence b: fuse + inject its whole context, draft the block,
    LM head.  Returns dict(fused, K, V, h, z, draft, margin, T)."""
    T = int(inputs.ctx_lens(w)[b])
    fused, K, V = ctx if ctx is not None else context(w, W, b, 0, T)
    ids = inputs.block_ids(w)[b].numpy()
    h = O.draft_block(K, V, T, ids, W, w, w.dtype == "bf16")
    z = O.lm_head(h, W["lm_head"])
    return dict(fused=fused, K=K, V=V, h=h, z=z, draft=O.argmax_lowest(z),
                margin=O.top2_margin(z), T=T)


def step_sequence(w: Workload, W, b, prefix, logits_row, u_row=None):
    """One timed oracle step of sequence b given its context K/V for positions
    [0, T-S) (`prefix` = (K, V) lists): fuse + inject the S newest rows, draft, LM head,
    verify.  Returns (draft, out_tokens, n_accepted, n_emitted)."""
    S = w.block_size
    T = int(inputs.ctx_lens(w)[b])
    _, k_new, v_new = context(w, W, b, T - S, T)
    K = [np.concatenate([prefix[0][l], k_new[l]]) for l in range(w.n_layers)]
    V = [np.concatenate([prefix[1][l], v_new[l]]) for l in range(w.n_layers)]
    r = draft_sequence(w, W, b, ctx=(None, K, V))
    if w.temperature > 0:
        out = O.verify_sample(r["draft"], r["z"], logits_row, u_row, w.temperature)
    else:
        out = O.verify_greedy(r["draft"], logits_row)
    return (r["draft"],) + tuple(out)


def draft_sequence_input(w: Workload, W, b):
    """The input-fusion variant of draft_sequence: the whole context of sequence b runs
    through the drafter's layer stack as input (causal), then the block is drafted.
    Returns dict(fused, K, V, h, z, draft, margin, T)."""
    T = int(inputs.ctx_lens(w)[b])
    x = np64(inputs.ctx_hidden(w, b, 0, T))
    ids = inputs.block_ids(w)[b].numpy()
    r = O.draft_step_input_fusion(x, T, ids, W, w, w.dtype == "bf16")
    r["T"] = T
    return r


def loop_weights(sw):
    """Host copies of the loop's drafter weights (with the target's embedding and LM
    head) and target weights."""
    tw = {k: v.float().numpy() for k, v in inputs.target_weights(sw).items()}
    dw = {n: inputs.weight(sw.drafter, n, s, k).float().numpy()
          for n, s, k in inputs.weight_specs(sw.drafter) if n not in ("embed", "lm_head")}
    dw["embed"], dw["lm_head"] = tw["embed"], tw["lm_head"]
    return dw, tw
