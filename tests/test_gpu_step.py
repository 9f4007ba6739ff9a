"""Parity of the whole CUDA step (inject -> draft -> LM head -> verify) with the fp64
oracle, element by element, on workloads the oracle finishes in seconds: the tiny fp32
workload at its full size, and bf16 shapes spanning several GEMM tiles, several context
pages with a ragged last page, permuted pages and a ragged vocabulary tail."""
import numpy as np
import pytest
import torch

from oracle import run as orun
from workload import configs, inputs

from gpu_helpers import check_drafts, check_greedy, gather_kv, head_parity, rel_err, tol

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny-f32": configs.TINY,
    "small-bf16-hd128": configs.small_bf16(),
    "small-bf16-hd64-g8": configs.small_bf16(
        name="small-bf16-hd64-g8", d_model=384, n_q_heads=16, n_kv_heads=2, head_dim=64,
        ffn_dim=384, vocab=2176, batch=3, ctx_range=(16, 120), seed=12),
    # batch 1 x block 16 rows (the 16-row projection tiles), two and one context splits
    "small-bf16-b1": configs.small_bf16(
        name="small-bf16-b1", batch=1, ctx_range=(150, 200), seed=14),
    "small-bf16-b1-1split": configs.small_bf16(
        name="small-bf16-b1-1split", batch=1, ctx_range=(40, 100), seed=15),
    "small-bf16-b5-s8": configs.small_bf16(
        name="small-bf16-b5-s8", block_size=8, batch=5, n_q_heads=4, n_kv_heads=2,
        ctx_range=(8, 70), vocab=1000, seed=13),
    # 96 and 320 block rows: the tcgen05 projection tiles (128 and 256 activation rows),
    # the second with a ragged 64-row second m-block; every tile split between CTAs
    "small-bf16-b6-tc128": configs.small_bf16(
        name="small-bf16-b6-tc128", batch=6, ctx_range=(20, 90), seed=16),
    "small-bf16-b20-tc256": configs.small_bf16(
        name="small-bf16-b20-tc256", batch=20, ctx_range=(16, 64), seed=17),
    # head_dim 64 with 96 and 80 block rows: attention on the tcgen05 kernel with 128 and
    # 64 query rows per kv head, ragged contexts over several splits and steps
    "small-bf16-hd64-g8-b6-tc": configs.small_bf16(
        name="small-bf16-hd64-g8-b6-tc", d_model=384, n_q_heads=16, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=6, ctx_range=(16, 250), seed=19),
    "small-bf16-hd64-g4-b5-tc": configs.small_bf16(
        name="small-bf16-hd64-g4-b5-tc", d_model=384, n_q_heads=8, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=5, ctx_range=(20, 180), seed=20),
    # one-page contexts (16 tokens: the split's single step holds the context page and
    # the block, so the tcgen05 key-split lanes of the step's second half see no valid
    # key) with 96 block rows at head_dim 128, and a mix of one- and two-page contexts
    # with 80 block rows at head_dim 64 (64 query rows per kv head)
    "small-bf16-b6-tc128-short": configs.small_bf16(
        name="small-bf16-b6-tc128-short", batch=6, ctx_range=(16, 16), seed=22),
    "small-bf16-hd64-g4-b5-short": configs.small_bf16(
        name="small-bf16-hd64-g4-b5-short", d_model=384, n_q_heads=8, n_kv_heads=2,
        head_dim=64, ffn_dim=384, vocab=2176, batch=5, ctx_range=(16, 24), seed=23),
    # 256 rows with K = 1024 and a 32000-token vocabulary: whole tiles per CTA as well
    "mid-bf16-b16-tc256": configs.small_bf16(
        name="mid-bf16-b16-tc256", d_model=1024, n_q_heads=8, n_kv_heads=2, head_dim=128,
        ffn_dim=2816, vocab=32000, batch=16, ctx_range=(16, 48), seed=18),
}


@pytest.fixture(scope="module")
def built():
    from block_diffusion_drafter_concat_gb300 import build
    build.build()


@pytest.mark.parametrize("name", list(SMALL))
def test_step_matches_oracle(built, name):
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = SMALL[name]
    r = StepRunner(w)
    W = orun.host_weights(w)
    seqs = [orun.draft_sequence(w, W, b) for b in range(w.batch)]
    drafts_o = np.stack([s["draft"] for s in seqs])
    r.plant(drafts_o)
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    t = tol(w)
    S = w.block_size
    hid = r.hidden.view(w.batch, S, -1)
    fused = r.fused.view(w.batch, S, -1)
    d_gpu = r.draft.cpu().numpy()
    out, nacc, nemit = r.out_tokens.cpu().numpy(), r.n_acc.cpu(), r.n_emit.cpu()
    checked = 0
    for b, s in enumerate(seqs):
        T = s["T"]
        assert rel_err(fused[b], s["fused"][T - S:T]) < t
        for l in range(w.n_layers):
            pos = np.arange(T)
            assert rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l]) < t
            assert rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l]) < t
        assert rel_err(hid[b], s["h"]) < t
        slack, _ = head_parity(d_gpu[b], hid[b], W["lm_head"], s["z"])
        check_drafts(d_gpu[b], s["draft"], s["margin"], slack)
        logits_row = r.logits[b].float().cpu().numpy()
        checked += check_greedy(out[b], nacc[b], nemit[b], d_gpu[b], logits_row)
    assert checked == w.batch


@pytest.mark.parametrize("name", ["small-bf16-hd128", "small-bf16-b1", "small-bf16-b20-tc256"])
def test_step_is_deterministic_and_graph_replay_matches(built, name):
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = SMALL[name]
    r = StepRunner(w)
    r.step()
    torch.cuda.synchronize()
    h1, d1 = r.hidden.clone(), r.draft.clone()
    r.step()
    torch.cuda.synchronize()
    assert torch.equal(h1, r.hidden) and torch.equal(d1, r.draft)
    r.capture()
    r.hidden.zero_()
    r.replay()
    torch.cuda.synchronize()
    assert torch.equal(h1, r.hidden) and torch.equal(d1, r.draft)
    assert r.drafter.device_error() == 0
