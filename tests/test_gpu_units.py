"""Per-entry-point GPU parity (LM head, fusion, verification) and device error paths,
each on oracle-side inputs drawn from the shared generator."""
import numpy as np
import pytest
import torch

import block_diffusion_drafter_concat_gb300 as pkg
from oracle import dflash_oracle as O
from oracle import run as orun
from workload import configs, inputs, synth

from gpu_helpers import check_drafts, check_sample, rel_err

pytestmark = pytest.mark.gpu

W_SMALL = configs.small_bf16()


@pytest.fixture(scope="module")
def small():
    from block_diffusion_drafter_concat_gb300 import build
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    build.build()
    return StepRunner(W_SMALL, prefill=False)


def hidden_rows(w, rows, name="h_test"):
    return synth.normal(w.seed, name, (rows, w.d_model), dtype=inputs.torch_dtype(w))


@pytest.mark.parametrize("rows", [1, 16, 37, 100, 130, 300])
def test_lm_head_argmax_stats(small, rows):
    w = W_SMALL
    h = hidden_rows(w, rows)
    tok = torch.empty(rows, dtype=torch.int32, device="cuda")
    mx = torch.empty(rows, dtype=torch.float32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    small.drafter.lm_head_argmax(h.cuda(), tok, small.ws, mx, lse, temperature=0.7)
    torch.cuda.synchronize()
    W = orun.host_weights(w)
    z = O.lm_head(orun.np64(h), W["lm_head"])
    check_drafts(tok.cpu().numpy(), O.argmax_lowest(z), O.top2_margin(z))
    assert rel_err(mx, z.max(axis=1)) < 1e-4
    zt = z / 0.7
    ref = zt.max(axis=1) + np.log(np.exp(zt - zt.max(axis=1, keepdims=True)).sum(axis=1))
    np.testing.assert_allclose(lse.cpu().numpy(), ref, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("rows", [1, 16, 37, 100, 300])
def test_lm_head_greedy_fused_argmax(small, rows):
    """Without lse the argmax is finished inside the projection (packed keys); two calls
    in a row also check that the keys and the CTA counter are left cleared."""
    w = W_SMALL
    W = orun.host_weights(w)
    for call in range(2):
        h = hidden_rows(w, rows, f"h_greedy{call}")
        tok = torch.empty(rows, dtype=torch.int32, device="cuda")
        mx = torch.empty(rows, dtype=torch.float32, device="cuda")
        small.drafter.lm_head_argmax(h.cuda(), tok, small.ws, mx, None, temperature=1.0)
        torch.cuda.synchronize()
        z = O.lm_head(orun.np64(h), W["lm_head"])
        check_drafts(tok.cpu().numpy(), O.argmax_lowest(z), O.top2_margin(z))
        assert rel_err(mx, z.max(axis=1)) < 1e-4
    assert small.drafter.device_error() == 0


@pytest.mark.parametrize("n", [1, 16, 45, 200, 513])
def test_fuse_features(small, n):
    w = W_SMALL
    x = synth.normal(w.seed, "x_fuse_test", (n, w.fuse_in), dtype=torch.bfloat16)
    out = torch.empty(n, w.d_model, dtype=torch.bfloat16, device="cuda")
    small.drafter.fuse_features(x.cuda(), out, small.ws)
    torch.cuda.synchronize()
    W = orun.host_weights(w)
    ref = O.fuse_features(orun.np64(x), W["w_fuse"], W["g_fuse"], w.rms_eps, True)
    assert rel_err(out, ref) < 2e-2


def test_verify_greedy_exact(small):
    w = W_SMALL
    B, S, V = 6, w.block_size, w.vocab
    g = torch.Generator().manual_seed(5)
    logits = (torch.randint(0, 6, (B, S, V), generator=g).float() - 3).to(torch.bfloat16)
    tgt = logits.float().argmax(-1)                        # lowest index on ties
    draft = tgt.clone()
    draft[1, 0] = (draft[1, 0] + 1) % V                    # mismatch at slot 0
    draft[2, 5] = (draft[2, 5] + 7) % V
    draft[4] = torch.randint(0, V, (S,), generator=g)
    draft = draft.to(torch.int32)
    out = torch.empty(B, S, dtype=torch.int32, device="cuda")
    na = torch.empty(B, dtype=torch.int32, device="cuda")
    ne = torch.empty(B, dtype=torch.int32, device="cuda")
    small.drafter.verify_greedy(draft.cuda(), logits.cuda(), out, na, ne, small.ws)
    torch.cuda.synchronize()
    for b in range(B):
        o, n, e = O.verify_greedy(draft[b].numpy(), logits[b].float().numpy())
        assert (int(na[b]), int(ne[b])) == (n, e)
        assert out[b].cpu().tolist() == list(o)
    assert int(ne[0]) == S and int(ne[1]) == 1 and int(na[2]) == 5


def test_verify_sample_matches_oracle(small):
    w = W_SMALL.scaled(temperature=1.0)
    B, S = 48, w.block_size
    rows = B * S
    h = hidden_rows(w, rows, "h_sample")
    W = orun.host_weights(w)
    z = O.lm_head(orun.np64(h), W["lm_head"])
    draft_o = O.argmax_lowest(z).reshape(B, S)
    margin = O.top2_margin(z).reshape(B, S)
    logits = synth.normal(w.seed, "logits_sample", (B, S, w.vocab), std=2.0,
                          dtype=torch.bfloat16)
    # plant partial agreement so acceptance walks go past slot 0
    mask = synth.uniform(w.seed, "plant_sample", (B, S)) < 0.6
    inputs.plant(w, logits, torch.as_tensor(draft_o), mask)
    u = synth.uniform(w.seed, "u_sample", (B, S, 2))
    hc = h.cuda()
    tok = torch.empty(rows, dtype=torch.int32, device="cuda")
    mx = torch.empty(rows, dtype=torch.float32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    small.drafter.lm_head_argmax(hc, tok, small.ws, mx, lse, temperature=1.0)
    out = torch.empty(B, S, dtype=torch.int32, device="cuda")
    na = torch.empty(B, dtype=torch.int32, device="cuda")
    ne = torch.empty(B, dtype=torch.int32, device="cuda")
    small.drafter.verify_sample(tok.view(B, S), hc, mx, lse, logits.cuda(), u.cuda(), 1.0, out,
                                na, ne, small.ws)
    torch.cuda.synchronize()
    assert small.drafter.device_error() == 0
    checked = 0
    lg = logits.float().numpy()
    zz = z.reshape(B, S, -1)
    d_gpu = tok.view(B, S).cpu().numpy()
    for b in range(B):
        # the head's drafts on identical input, then the walk over those drafts
        check_drafts(d_gpu[b], draft_o[b], margin[b])
        checked += check_sample(out[b].cpu().numpy(), na[b], ne[b], d_gpu[b], zz[b], lg[b],
                                u[b].numpy(), 1.0)
    assert checked >= B // 2


def test_device_errors_are_reported_not_trapped(small):
    r = small
    w = r.w
    r.prefill()
    d = r.drafter
    # block token id out of range
    bad_ids = r.block_ids.clone()
    bad_ids[0, 0] = w.vocab + 3
    d.draft_block(bad_ids, r.ctx_lens, r.page_table, r.cache, r.hidden, r.ws)
    assert d.device_error() == 1
    d.workspace_init(r.ws)
    # context longer than the page table allows
    bad_lens = r.ctx_lens.clone()
    bad_lens[0] = w.max_pages * 16 + 1
    d.draft_block(r.block_ids, bad_lens, r.page_table, r.cache, r.hidden, r.ws)
    assert d.device_error() in (1, 2)
    d.workspace_init(r.ws)
    # a page id outside the pool
    bad_table = r.page_table.clone()
    bad_table[0, 0] = r.cache.num_pages + 5
    d.draft_block(r.block_ids, r.ctx_lens, bad_table, r.cache, r.hidden, r.ws)
    assert d.device_error() == 1
    d.workspace_init(r.ws)
    # the path still works afterwards
    r.step()
    torch.cuda.synchronize()
    assert d.device_error() == 0


def test_device_errors_on_the_tcgen05_paths():
    """The same device checks on blocks of 96 rows with head_dim 64: projections and
    attention on the tcgen05 kernels (slot, page-id and position checks)."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = configs.small_bf16(name="err-hd64-b6", d_model=384, n_q_heads=16, n_kv_heads=2,
                           head_dim=64, ffn_dim=384, vocab=2176, batch=6,
                           ctx_range=(40, 200), seed=21)
    r = StepRunner(w)
    d = r.drafter
    bad_table = r.page_table.clone()
    bad_table[2, 1] = r.cache.num_pages + 7
    d.draft_block(r.block_ids, r.ctx_lens, bad_table, r.cache, r.hidden, r.ws)
    assert d.device_error() == 1
    d.workspace_init(r.ws)
    bad_slots = r.slots.clone()
    bad_slots[50] = -4
    d.inject_kv(r.positions, bad_slots, r.cache, r.ws, x_cat=r.x_step)
    assert d.device_error() == 1
    d.workspace_init(r.ws)
    bad_pos = r.positions.clone()
    bad_pos[17] = w.max_position + 2
    d.inject_kv(bad_pos, r.slots, r.cache, r.ws, x_cat=r.x_step)
    assert d.device_error() == 2
    d.workspace_init(r.ws)
    r.step()
    torch.cuda.synchronize()
    assert d.device_error() == 0


def test_host_validation_statuses(small):
    r = small
    d = r.drafter
    tiny_ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.DFlashError) as e:
        d.draft_block(r.block_ids, r.ctx_lens, r.page_table, r.cache, r.hidden, tiny_ws)
    assert e.value.status == pkg.EWORKSPACE
    with pytest.raises(pkg.DFlashError) as e:
        d.lm_head_argmax(r.hidden[:, 1:], r.draft.view(-1), r.ws)   # misaligned rows
    assert e.value.status == pkg.EINVAL


# 32 block rows (mma.sync projections, stream-K with split tiles at these sizes) and 320
# rows with an 80000-token vocabulary (the tcgen05 LM head's 1250 tiles are planned as
# stream-K ranges, which split tiles between CTAs)
TIMEOUT_WORKLOADS = {
    "small-bf16-hd128": configs.PARITY_SMALL["small-bf16-hd128"],
    "timeout-tc256-v80k": configs.small_bf16(name="timeout-tc256-v80k", batch=20, vocab=80000,
                                             ctx_range=(16, 64), seed=24),
    # 96 rows: the tcgen05 kernel's 128-row tiles, whose split finish counts after publishing
    "timeout-tc128-v80k": configs.small_bf16(name="timeout-tc128-v80k", batch=6, vocab=80000,
                                             ctx_range=(16, 64), seed=25),
}


@pytest.mark.parametrize("name", list(TIMEOUT_WORKLOADS))
def test_forced_wait_timeout_is_reported_and_recovered(name):
    """The bounded on-device waits: with the test hook on, every split-tile finisher
    (mma.sync or tcgen05 projections) waits for one piece more than can arrive, gives up
    after 10 ms and reports DFLASH_DEV_TIMEOUT instead of hanging; after the hook is off
    and the workspace re-initialised, the next step is clean and bit-identical to one
    made before."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    r = StepRunner(TIMEOUT_WORKLOADS[name])
    d = r.drafter
    r.step()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    h_ref, d_ref = r.hidden.clone(), r.draft.clone()
    d.test_force_timeout(True)
    try:
        r.step()
        assert d.device_error() == 3
    finally:
        d.test_force_timeout(False)
    d.workspace_init(r.ws)
    r.hidden.zero_()
    r.step()
    torch.cuda.synchronize()
    assert d.device_error() == 0
    assert torch.equal(r.hidden, h_ref) and torch.equal(r.draft, d_ref)
