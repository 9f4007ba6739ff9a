"""Named synthetic tensors of a workload (weights, context, logits, uniforms).

Every tensor is drawn from :mod:`workload.synth` under a fixed name, so the host copy
used by the oracle and the device copy used by the CUDA path are the same numbers.
Matrices are N(0, weight_std) in the ``[out, in]`` convention, RMSNorm gains are
1 + N(0, gain_std), target hidden features N(0, hidden_std), verify logits
N(0, logit_std); bf16 workloads round every drawn value to bf16 once.
Nothing here computes any part of the drafter.
"""
from __future__ import annotations

import torch

from . import synth
from .configs import Workload


def torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def weight_specs(w: Workload):
    """(name, shape, kind) for every drafter weight, in a fixed order."""
    d, F, V = w.d_model, w.ffn_dim, w.vocab
    specs = [("w_fuse", (d, w.fuse_in), "mat"), ("g_fuse", (d,), "gain")]
    for l in range(w.n_layers):
        specs += [
            (f"l{l}.g_attn", (d,), "gain"),
            (f"l{l}.w_q", (w.q_width, d), "mat"),
            (f"l{l}.w_k", (w.kv_width, d), "mat"),
            (f"l{l}.w_v", (w.kv_width, d), "mat"),
            (f"l{l}.w_o", (d, w.q_width), "mat"),
            (f"l{l}.g_mlp", (d,), "gain"),
            (f"l{l}.w_gate", (F, d), "mat"),
            (f"l{l}.w_up", (F, d), "mat"),
            (f"l{l}.w_down", (d, F), "mat"),
        ]
    specs += [("g_final", (d,), "gain"), ("embed", (V, d), "mat"), ("lm_head", (V, d), "mat")]
    return specs


def weight(w: Workload, name, shape, kind, device="cpu", dtype=None):
    dtype = dtype or torch_dtype(w)
    if kind == "gain":
        return synth.normal(w.seed, name, shape, std=w.gain_std, mean=1.0, dtype=dtype,
                            device=device)
    return synth.normal(w.seed, name, shape, std=w.weight_std, dtype=dtype, device=device)


def weights(w: Workload, device="cpu"):
    return {n: weight(w, n, s, k, device) for n, s, k in weight_specs(w)}


def ctx_lens(w: Workload) -> torch.Tensor:
    """T_b per sequence (context length after this step's injection), int64 host."""
    if w.ctx_range is None:
        return torch.full((w.batch,), w.ctx_len, dtype=torch.int64)
    lo, hi = w.ctx_range
    return synth.integers(w.sseed, "ctx_len", (w.batch,), lo, hi)


def page_table(w: Workload, lens=None):
    """(page_table [B, max_pages] int32 with -1 past each sequence, num_pages).

    Pages are handed out in a seeded random order when ``permute_pages`` is set, so
    logically adjacent context pages sit far apart in the pool."""
    lens = ctx_lens(w) if lens is None else lens
    npg = [-(-int(t) // w.page_size) for t in lens]
    total = sum(npg)
    order = synth.permutation(w.sseed, "pages", total) if w.permute_pages \
        else torch.arange(total)
    table = torch.full((w.batch, w.max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npg):
        table[b, :n] = order[off:off + n].to(torch.int32)
        off += n
    return table, total


def slots_for(w: Workload, table, b, positions):
    """Cache slot (page * page_size + offset) of context positions of sequence b."""
    positions = torch.as_tensor(positions, dtype=torch.int64)
    pages = table[b].to(torch.int64)[positions // w.page_size]
    return pages * w.page_size + positions % w.page_size


def ctx_hidden(w: Workload, b, p0, p1, device="cpu"):
    """Concatenated target hidden features X_cat of sequence b, positions [p0, p1):
    ``[p1-p0, n_target_layers*target_width]``, target layer l in columns
    [l*target_width, (l+1)*target_width)."""
    shape = (w.batch * w.max_ctx, w.fuse_in)
    r0 = b * w.max_ctx + p0
    return synth.normal(w.sseed, "x_ctx", shape, std=w.hidden_std, dtype=torch_dtype(w),
                        device=device, rows=(r0, r0 + (p1 - p0)))


def block_ids(w: Workload):
    return torch.full((w.batch, w.block_size), w.mask_id, dtype=torch.int32)


def logits_noise(w: Workload, b0=0, b1=None, device="cpu"):
    """Unplanted target verify logits of sequences [b0, b1): [b1-b0, S, V]."""
    b1 = w.batch if b1 is None else b1
    shape = (w.batch * w.block_size, w.vocab)
    z = synth.normal(w.sseed, "logits", shape, std=w.logit_std, dtype=torch_dtype(w),
                     device=device, rows=(b0 * w.block_size, b1 * w.block_size))
    return z.view(b1 - b0, w.block_size, w.vocab)


def plant_mask(w: Workload):
    """[B, S] bool: positions where the target agrees with the draft."""
    return synth.uniform(w.sseed, "plant", (w.batch, w.block_size)) < w.agree_p


def decoy_drafts(w: Workload):
    return synth.integers(w.sseed, "decoy", (w.batch, w.block_size), 0, w.vocab - 1)


def plant(w: Workload, logits, drafts, mask):
    """Raise logit[draft] to (row max + 1) at the masked positions, in place.

    logits [b, S, V] (any device), drafts [b, S] int, mask [b, S] bool (host)."""
    dev = logits.device
    drafts = torch.as_tensor(drafts, dtype=torch.int64).to(dev)
    mask = torch.as_tensor(mask).to(dev)
    top = logits.float().amax(dim=-1) + 1.0
    cur = logits.gather(-1, drafts[..., None])[..., 0]
    new = torch.where(mask, top.to(logits.dtype), cur)
    logits.scatter_(-1, drafts[..., None], new[..., None])
    return logits


def uniforms(w: Workload, device="cpu"):
    """[B, S, 2] fp32: [..., 0] acceptance test, [..., 1] residual draw."""
    return synth.uniform(w.sseed, "uniforms", (w.batch, w.block_size, 2), device=device)


# ------------------------------------------------------------- speculative loop
def target_weights(sw, device="cpu"):
    """The loop's target: every drafter layer weight name, the final gain, embedding
    and LM head, from the target's own seed (no fusion weights)."""
    wt = sw.target
    return {n: weight(wt, n, s, k, device) for n, s, k in weight_specs(wt)
            if n not in ("w_fuse", "g_fuse")}


def loop_drafter_weights(sw, target_w, device="cpu"):
    """The drafter's own weights with the target's embedding and LM head (reused)."""
    w = sw.drafter
    out = {n: weight(w, n, s, k, device) for n, s, k in weight_specs(w)
           if n not in ("embed", "lm_head")}
    out["embed"], out["lm_head"] = target_w["embed"], target_w["lm_head"]
    return out


def prompt_tokens(sw):
    """[B, prompt_len] int64 random prompt tokens (host)."""
    w = sw.drafter
    return synth.integers(w.seed, "prompt", (w.batch, sw.prompt_len), 0, w.vocab - 1)


def loop_uniforms(sw, device="cpu"):
    """[steps, B, S] fp32 uniforms of the planted agreement, one per verified slot."""
    w = sw.drafter
    return synth.uniform(w.seed, "plant_loop", (sw.steps, w.batch, w.block_size), device=device)
