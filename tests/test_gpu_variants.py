"""Parity of the two rows beyond the single step: the input-fusion variant of the
drafter (dflash_inject_inputs: the context runs through the layer stack, causally,
before the block is drafted) and the greedy speculative loop with a random target
(dflash_target_forward, dflash_spec_step), each against the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from oracle import run as orun
from workload import configs, inputs

from gpu_helpers import (capped_draft_check, check_greedy, gather_kv, head_parity, rel_err,
                         tol)
from parity_plan import MIN_CHECKED, report

pytestmark = pytest.mark.gpu

INPUT_FUSION = ["tiny-f32", "small-bf16-hd128", "small-bf16-b1", "small-bf16-hd64-g8-b6-tc",
                "small-bf16-b20-tc256", "qwen3-8b-shaped-b1"]


@pytest.fixture(scope="module")
def built():
    from block_diffusion_drafter_concat_gb300 import build
    build.build()


def _workload(name):
    return configs.PARITY_SMALL.get(name) or configs.BY_NAME[name]


@pytest.mark.parametrize("name", INPUT_FUSION)
def test_input_fusion_step_matches_oracle(built, name):
    """Cache K/V of every layer (each the output of the causal layer stack over the
    context), the final hidden state, drafts (capped slack) and verification."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = _workload(name)
    r = StepRunner(w, variant="input")
    W = orun.host_weights(w)
    seqs = [orun.draft_sequence_input(w, W, b) for b in range(w.batch)]
    r.plant(np.stack([s["draft"] for s in seqs]))
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    t, S = tol(w), w.block_size
    hid = r.hidden.view(w.batch, S, -1)
    d_gpu = r.draft.cpu().numpy()
    rows_checked = rows_out = 0
    dz_max = 0.0
    for b, s in enumerate(seqs):
        T = s["T"]
        assert rel_err(r.fused.view(w.batch, S, -1)[b], s["fused"][T - S:T]) < t
        pos = np.arange(T) if T <= 4096 else np.arange(0, T, 7)
        for l in range(w.n_layers):
            assert rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l][pos]) < t, l
            assert rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l][pos]) < t, l
        assert rel_err(hid[b], s["h"]) < t
        dz, _ = head_parity(d_gpu[b], hid[b], W["lm_head"], s["z"])
        c, o = capped_draft_check("input:" + name, d_gpu[b], s["draft"], s["margin"], dz)
        rows_checked += c
        rows_out += o
        dz_max = max(dz_max, float(dz.max()))
        assert check_greedy(r.out_tokens[b].cpu().numpy(), r.n_acc[b].cpu(), r.n_emit[b].cpu(),
                            d_gpu[b], r.logits[b].float().cpu().numpy())
    report("input:" + name, dict(test="input-fusion step", dz_max=dz_max,
                                 rows_checked=rows_checked, rows_left_out=rows_out))
    assert rows_checked >= MIN_CHECKED * (rows_checked + rows_out)


def test_input_fusion_differs_from_kv_injection(built):
    """The two variants put different K/V into the cache beyond layer 0 (the input-fusion
    context is mixed by attention before each deeper layer)."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = configs.PARITY_SMALL["small-bf16-hd128"]
    a, b = StepRunner(w), StepRunner(w, variant="input")
    a.step()
    b.step()
    torch.cuda.synchronize()
    assert not torch.equal(a.cache.k[1], b.cache.k[1])


# ------------------------------------------------------------------ speculative loop
# Decisions are compared where the oracle's top-2 margin is at least THR: fp32 deviations
# are ~1e-5; the small bf16 workloads' rounding-flip logit changes stay below 0.02
# (their stored caps), so 0.05 leaves a factor of more than two.
THR = {"f32": 1e-2, "bf16": 5e-2}


def _run_loop(sw, plant):
    from block_diffusion_drafter_concat_gb300.spec import SpecRunner
    r = SpecRunner(sw, plant=plant)
    r.prefill()
    hist = []
    for _ in range(sw.steps):
        r.step()
        torch.cuda.synchronize()
        hist.append(dict(drafts=r.drafts.cpu().numpy().copy(),
                         n_emit=r.n_emitted.cpu().numpy().copy()))
    assert r.drafter.device_error() == 0 and r.target.device_error() == 0
    gen = r.generated.cpu().numpy()
    ng = r.n_generated.cpu().numpy()
    ctx = r.ctx_lens.cpu().numpy()
    return r, hist, gen, ng, ctx


def _walk(block, d_gpu, em_gpu, thr):
    """The verification walk over the oracle's (planted) block logits and the GPU's
    drafts, taking the GPU's token at rows whose top-2 margin is below thr (after
    checking that it is within thr of the row's maximum).  Returns (emitted tokens,
    near-tie rows met)."""
    S = len(d_gpu)
    out, near = [], 0
    for i in range(S):
        row = block[i]
        if O.top2_margin(row) >= thr:
            t = int(O.argmax_lowest(row))
        else:
            near += 1
            assert i < len(em_gpu), (i, em_gpu)
            t = int(em_gpu[i])
            assert row[t] >= row.max() - thr, (i, t, row[t], row.max())
        out.append(t)
        if i == S - 1 or int(d_gpu[i + 1]) != t:
            return out, near
    return out, near


@pytest.mark.parametrize("name", ["spec-tiny-f32", "spec-small-bf16"])
def test_spec_loop_matches_oracle(built, name):
    """Every step of every sequence, teacher-forced on the GPU's own history: the GPU's
    drafts are the oracle drafter's argmax (or within THR of it at a near tie), and the
    verification walk of those drafts over the oracle target's planted logits gives the
    GPU's accepted length and emitted tokens exactly (at a target row within THR of a
    tie the GPU's token is taken once checked to be a valid near-maximum)."""
    sw = configs.SPEC[name]
    w = sw.drafter
    bf16 = w.dtype == "bf16"
    thr = THR[w.dtype]
    r, hist, gen, ng, ctx = _run_loop(sw, plant=True)
    S = w.block_size
    Wd, Wt = orun.loop_weights(sw)
    u = inputs.loop_uniforms(sw).numpy()
    prompt = inputs.prompt_tokens(sw).numpy()
    near_drafts = near_rows = emitted_total = 0
    for b in range(w.batch):
        seq = list(prompt[b])
        off = 0
        for k, hk in enumerate(hist):
            d_gpu = hk["drafts"][b]
            ne = int(hk["n_emit"][b])
            assert 1 <= ne <= S
            em_gpu = gen[b, off:off + ne]
            fn = O.dflash_drafter(Wd, w, bf16, mask_id=w.mask_id)
            feats, _ = O.target_forward(np.asarray(seq[:-1]), Wt, sw.target, bf16, sw.tap_layers)
            d_o = fn(np.asarray(seq), feats)
            z = fn.calls[-1]
            for i in range(1, S):
                if d_gpu[i] != d_o[i]:
                    near_drafts += 1
                    assert O.top2_margin(z[i]) < thr and z[i][d_gpu[i]] >= z[i].max() - thr, \
                        (b, k, i, d_gpu[i], d_o[i])
            _, _, _, block = O.spec_step(np.asarray(seq), lambda c, f: d_gpu, Wt, sw.target,
                                         bf16, sw.tap_layers, S, u[k, b], sw.plant_p)
            want, near = _walk(block, d_gpu, em_gpu, thr)
            near_rows += near
            assert list(map(int, em_gpu)) == want, (b, k, em_gpu, want)
            seq += want
            off += ne
            emitted_total += ne
        assert ng[b] == off and ctx[b] == sw.prompt_len - 1 + off
    report(name, dict(test="spec loop", steps=w.batch * sw.steps, near_tie_drafts=near_drafts,
                      near_tie_target_rows=near_rows,
                      mean_emitted=emitted_total / (w.batch * sw.steps)))
    assert emitted_total > w.batch * sw.steps      # planting makes drafts accepted


@pytest.mark.parametrize("name", ["spec-tiny-f32", "spec-small-bf16"])
def test_spec_loop_without_planting_is_the_targets_greedy_decoding(built, name):
    """Greedy speculative decoding is lossless: without planting, every token the GPU
    loop emits is the oracle target's autoregressive greedy choice given the tokens
    before it (or, where the oracle's top-2 margin is below THR, one within THR of the
    maximum)."""
    sw = configs.SPEC[name]
    w = sw.drafter
    bf16 = w.dtype == "bf16"
    thr = THR[w.dtype]
    r, hist, gen, ng, ctx = _run_loop(sw, plant=False)
    _, Wt = orun.loop_weights(sw)
    prompt = inputs.prompt_tokens(sw).numpy()
    clear = near = 0
    for b in range(w.batch):
        seq = list(prompt[b])
        for j in range(int(ng[b])):
            _, logits = O.target_forward(np.asarray(seq), Wt, sw.target, bf16, ())
            last, t = logits[-1], int(gen[b, j])
            if O.top2_margin(last) >= thr:
                assert t == int(O.argmax_lowest(last)), (b, j)
                clear += 1
            else:
                assert last[t] >= last.max() - thr, (b, j)
                near += 1
            seq.append(t)
    report(name, dict(test="spec loop lossless", tokens_clear=clear, tokens_near_tie=near))
    assert clear + near >= w.batch * sw.steps and clear >= near
