"""Parity at the full sizes of the four large workloads (and their one-layer variants),
in the launch configuration the benchmark times.

Every sequence of the batch: the drafted tokens are the oracle's LM-head argmax of the
GPU's own final hidden state (exact outside 1e-2 margins), and the verification result
is the oracle's walk over those drafts and the same target logits (greedy: bit-exact;
temperature 1: exact acceptance decisions and a valid residual draw).

A seeded sample of sequences (the shortest, the longest and evenly spaced context
lengths between): fused features and injected K/V of the step rows, K/V of sampled
earlier context positions, the final hidden state, and the drafted tokens against the
oracle's own drafts with the slack capped by the oracle-derived constant of the
workload (tests/parity_plan.py).

The verify logits are planted from the oracle's drafts on the sampled sequences and
from the GPU's first-step drafts on the others (the step is then run again on the same
inputs), so every verification walk goes past its first slot.
"""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from oracle import run as orun
from workload import configs, inputs

from gpu_helpers import (MARGIN, capped_draft_check, check_drafts, check_greedy, check_sample,
                         gather_kv, head_parity, rel_err, tol)
from parity_plan import MIN_CHECKED, report, sampled_sequences

pytestmark = pytest.mark.gpu

FULL = ["qwen3-8b-shaped-b1", "qwen3-8b-shaped-b32-ragged", "llama-3.1-8b-shaped-b8",
        "gpt-oss-120b-shaped-b64-t1"]


@pytest.fixture(scope="module")
def built():
    from block_diffusion_drafter_concat_gb300 import build
    build.build()


def run_full(w, bs, W, seqs):
    """The benchmark's step on workload w, with the verify logits planted from the
    oracle's drafts on the sequences in `bs` and the GPU's own drafts elsewhere."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    r = StepRunner(w)
    r.step()
    torch.cuda.synchronize()
    drafts = r.draft.cpu().clone()
    for b in bs:
        drafts[b] = torch.as_tensor(seqs[b]["draft"])
    r.plant(drafts)
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    return r


def all_sequences(name, w, r, W):
    """Head and verification parity on every sequence; returns the oracle's logits of
    the GPU's hidden state (for the sampled checks)."""
    S = w.block_size
    hid = r.hidden.float().cpu().numpy().astype(np.float64)
    d_gpu = r.draft.cpu().numpy()
    _, zg = head_parity(d_gpu.reshape(-1), hid, W["lm_head"])
    zg = zg.reshape(w.batch, S, -1)
    out, nacc, nemit = r.out_tokens.cpu().numpy(), r.n_acc.cpu(), r.n_emit.cpu()
    unambiguous = 0
    for b in range(w.batch):
        lg = r.logits[b].float().cpu().numpy()
        if w.temperature > 0:
            # the drafter distribution of the GPU's drafts: the oracle's LM head on the
            # GPU's hidden state
            unambiguous += check_sample(out[b], nacc[b], nemit[b], d_gpu[b], zg[b], lg,
                                        r.uniforms[b].cpu().numpy(), w.temperature)
        else:
            unambiguous += check_greedy(out[b], nacc[b], nemit[b], d_gpu[b], lg)
    # greedy walks are always compared; temperature-1 walks that meet an acceptance
    # ratio within 1e-3 of their uniform are left out
    assert unambiguous >= (w.batch if w.temperature == 0 else (w.batch + 1) // 2), unambiguous
    return zg, unambiguous


def sampled_parity(name, w, r, W, seqs, bs, zg, plain_margin):
    S, t = w.block_size, tol(w)
    hid = r.hidden.view(w.batch, S, -1)
    fused = r.fused.view(w.batch, S, -1)
    d_gpu = r.draft.cpu().numpy()
    rng = np.random.default_rng(0)
    rows_checked = rows_out = 0
    dz_max = 0.0
    for b in bs:
        s = seqs[b]
        T = s["T"]
        errs = {"fused": rel_err(fused[b], s["fused"][T - S:T]), "h": rel_err(hid[b], s["h"])}
        pos = np.concatenate([np.arange(T - S, T), rng.choice(T - S, 48, replace=False)])
        for l in range(w.n_layers):
            errs[f"k{l}"] = rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l][pos])
            errs[f"v{l}"] = rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l][pos])
        assert max(errs.values()) < t, (b, errs)
        dz = np.abs(zg[b] - s["z"]).max(axis=-1)
        dz_max = max(dz_max, float(dz.max()))
        if plain_margin:
            low = check_drafts(d_gpu[b], s["draft"], s["margin"])
            c, o = int((~low).sum()), int(low.sum())
        else:
            c, o = capped_draft_check(name, d_gpu[b], s["draft"], s["margin"], dz)
        rows_checked += c
        rows_out += o
    rec = dict(test="full", sequences=list(map(int, bs)), dz_max=dz_max,
               rows_checked=rows_checked, rows_left_out=rows_out,
               margin="1e-2" if plain_margin else "max(1e-2, 2 dz), dz capped")
    return rec


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(built, name):
    w = configs.BY_NAME[name]
    bs = sampled_sequences(inputs.ctx_lens(w).numpy())
    W = orun.host_weights(w)
    seqs = {b: orun.draft_sequence(w, W, b) for b in bs}
    r = run_full(w, bs, W, seqs)
    zg, unamb = all_sequences(name, w, r, W)
    rec = sampled_parity(name, w, r, W, seqs, bs, zg, plain_margin=False)
    rec["verify_walks_compared"] = int(unamb)
    report(name, rec)
    print(name, rec)
    assert rec["rows_checked"] >= MIN_CHECKED * (rec["rows_checked"] + rec["rows_left_out"])
    del r
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", list(configs.ONE_LAYER))
def test_one_layer_full_width_plain_margin(built, name):
    """Full-width shapes with a single drafter layer (fewer compounding rounding
    points): drafts compared at the plain 1e-2 top-2 margin on four sampled sequences."""
    w = configs.ONE_LAYER[name]
    bs = sampled_sequences(inputs.ctx_lens(w).numpy(), k=4)
    W = orun.host_weights(w)
    seqs = {b: orun.draft_sequence(w, W, b) for b in bs}
    r = run_full(w, bs, W, seqs)
    zg, unamb = all_sequences(name, w, r, W)
    rec = sampled_parity(name, w, r, W, seqs, bs, zg, plain_margin=True)
    rec["verify_walks_compared"] = int(unamb)
    report(name, rec)
    print(name, rec)
    assert MARGIN == 1e-2
    del r
    torch.cuda.empty_cache()
