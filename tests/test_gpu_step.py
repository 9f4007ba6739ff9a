"""Parity of the whole CUDA step (inject -> draft -> LM head -> verify) with the fp64
oracle, element by element, on workloads the oracle finishes in seconds: the tiny fp32
workload at its full size, and bf16 shapes spanning several GEMM tiles, several context
pages with a ragged last page, permuted pages and a ragged vocabulary tail."""
import numpy as np
import pytest
import torch

from oracle import run as orun
from workload import configs, inputs

from gpu_helpers import (capped_draft_check, check_greedy, gather_kv, head_parity,
                         rel_err, tol)
from parity_plan import MIN_CHECKED, report

pytestmark = pytest.mark.gpu

SMALL = configs.PARITY_SMALL


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
    rows_checked = rows_out = 0
    dz_max = 0.0
    for b, s in enumerate(seqs):
        T = s["T"]
        assert rel_err(fused[b], s["fused"][T - S:T]) < t
        for l in range(w.n_layers):
            pos = np.arange(T)
            assert rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l]) < t
            assert rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l]) < t
        assert rel_err(hid[b], s["h"]) < t
        dz, _ = head_parity(d_gpu[b], hid[b], W["lm_head"], s["z"])
        c, o = capped_draft_check(name, d_gpu[b], s["draft"], s["margin"], dz)
        rows_checked += c
        rows_out += o
        dz_max = max(dz_max, float(dz.max()))
        logits_row = r.logits[b].float().cpu().numpy()
        checked += check_greedy(out[b], nacc[b], nemit[b], d_gpu[b], logits_row)
    assert checked == w.batch
    report(name, dict(test="step", dz_max=dz_max, rows_checked=rows_checked,
                      rows_left_out=rows_out))
    assert rows_checked >= MIN_CHECKED * (rows_checked + rows_out)


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
