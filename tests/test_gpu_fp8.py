"""FP8 weight streaming on the GPU: the packed form written by dflash_pack_fp8 is the
oracle quantizer's, code for code and scale for scale; a step whose projections stream
those packed weights matches the fp64 oracle run with the same dequantized weights
(the parity bars of the bf16 step); and how far FP8 weights move the drafts from the
bf16 drafter's is reported."""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from oracle import run as orun
from workload import configs, inputs, synth

from gpu_helpers import capped_draft_check, check_greedy, gather_kv, head_parity, rel_err
from parity_plan import MIN_CHECKED, report, sampled_sequences

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def built():
    from block_diffusion_drafter_concat_gb300 import build
    build.build()


@pytest.mark.parametrize("rows,cols", [(1, 16), (7, 100), (128, 512), (300, 1000), (64, 4096)])
def test_packing_is_the_oracle_quantizer(built, rows, cols):
    import block_diffusion_drafter_concat_gb300 as pkg
    w = synth.normal(5, f"pack{rows}x{cols}", (rows, cols), std=0.02, dtype=torch.bfloat16)
    if rows > 3:
        w[2] = 0                                   # an all-zero row
        w[3, cols // 2] = 7.5                      # an outlier
    packed = pkg.pack_fp8(w.cuda())
    torch.cuda.synchronize()
    codes, scales = pkg.unpack_fp8(packed, rows, cols)
    q, s = O.quantize_rows_fp8(w.float().numpy())
    got = codes.cpu().contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, q)
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.float64), s)
    ld = (cols + 15) // 16 * 16
    if ld > cols:                                  # row padding is zero
        pad = packed[:rows * ld].view(rows, ld)[:, cols:]
        assert int(pad.to(torch.int32).sum()) == 0


@pytest.mark.parametrize("name", [n for n in configs.FP8 if not n.startswith("qwen")])
def test_fp8_step_matches_oracle(built, name):
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = configs.FP8[name]
    r = StepRunner(w)
    W = orun.host_weights(w)                       # dequantized FP8 projections
    seqs = [orun.draft_sequence(w, W, b) for b in range(w.batch)]
    r.plant(np.stack([s["draft"] for s in seqs]))
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    S = w.block_size
    hid = r.hidden.view(w.batch, S, -1)
    d_gpu = r.draft.cpu().numpy()
    rows_checked = rows_out = 0
    dz_max = 0.0
    for b, s in enumerate(seqs):
        T = s["T"]
        assert rel_err(r.fused.view(w.batch, S, -1)[b], s["fused"][T - S:T]) < 2e-2
        pos = np.arange(T)
        for l in range(w.n_layers):
            assert rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l]) < 2e-2
            assert rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l]) < 2e-2
        assert rel_err(hid[b], s["h"]) < 2e-2
        dz, _ = head_parity(d_gpu[b], hid[b], W["lm_head"], s["z"])
        c, o = capped_draft_check(name, d_gpu[b], s["draft"], s["margin"], dz)
        rows_checked += c
        rows_out += o
        dz_max = max(dz_max, float(dz.max()))
        assert check_greedy(r.out_tokens[b].cpu().numpy(), r.n_acc[b].cpu(), r.n_emit[b].cpu(),
                            d_gpu[b], r.logits[b].float().cpu().numpy())
    report(name, dict(test="fp8 step", dz_max=dz_max, rows_checked=rows_checked,
                      rows_left_out=rows_out))
    assert rows_checked >= MIN_CHECKED * (rows_checked + rows_out)


def test_fp8_full_size_batch1(built):
    """The Qwen3-8B-shaped batch-1 step with FP8 weights: fused features, K/V of the
    step rows and of sampled earlier positions, final hidden state, drafts (capped
    slack) and verification; plus the agreement of its drafts with the bf16 drafter's
    (quantization, not kernel error: reported)."""
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    name = "qwen3-8b-shaped-b1-fp8"
    w = configs.FP8[name]
    W = orun.host_weights(w)
    s = orun.draft_sequence(w, W, 0)
    r = StepRunner(w)
    r.plant(torch.as_tensor(s["draft"])[None])
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    S, T = w.block_size, s["T"]
    rng = np.random.default_rng(0)
    pos = np.concatenate([np.arange(T - S, T), rng.choice(T - S, 48, replace=False)])
    errs = {"fused": rel_err(r.fused, s["fused"][T - S:T]), "h": rel_err(r.hidden, s["h"])}
    for l in range(w.n_layers):
        errs[f"k{l}"] = rel_err(gather_kv(r.cache.k[l], r.table_host, 0, pos), s["K"][l][pos])
        errs[f"v{l}"] = rel_err(gather_kv(r.cache.v[l], r.table_host, 0, pos), s["V"][l][pos])
    assert max(errs.values()) < 2e-2, errs
    d_gpu = r.draft.cpu().numpy()[0]
    dz, _ = head_parity(d_gpu, r.hidden, W["lm_head"], s["z"])
    c, o = capped_draft_check(name, d_gpu, s["draft"], s["margin"], dz)
    assert check_greedy(r.out_tokens[0].cpu().numpy(), r.n_acc[0].cpu(), r.n_emit[0].cpu(),
                        d_gpu, r.logits[0].float().cpu().numpy())
    bf = orun.draft_sequence(configs.QWEN3_8B_B1, orun.host_weights(configs.QWEN3_8B_B1), 0)
    report(name, dict(test="fp8 full", dz_max=float(dz.max()), rows_checked=c, rows_left_out=o,
                      drafts_equal_to_bf16_drafter=int((d_gpu == bf["draft"]).sum()),
                      h_rel_err_vs_bf16=rel_err(r.hidden, bf["h"])))
    assert c >= MIN_CHECKED * (c + o)
