"""Parity at the full sizes of the four large workloads, in the launch configuration the
benchmark times, on sampled sequences the oracle computes one by one: fused features
and injected K/V of the step rows, K/V of sampled earlier context positions, the final
hidden state, the drafted tokens and the verification result."""
import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O
from oracle import run as orun
from workload import configs, inputs

from gpu_helpers import (check_drafts, check_greedy, check_sample, gather_kv, head_parity,
                         rel_err, tol)

pytestmark = pytest.mark.gpu


def sampled(w):
    lens = inputs.ctx_lens(w)
    if w.ctx_range:
        return sorted({int(lens.argmin()), int(lens.argmax())})
    return sorted({0, w.batch - 1})


@pytest.fixture(scope="module")
def built():
    from block_diffusion_drafter_concat_gb300 import build
    build.build()


@pytest.mark.parametrize("name", ["qwen3-8b-shaped-b1", "qwen3-8b-shaped-b32-ragged",
                                  "llama-3.1-8b-shaped-b8", "gpt-oss-120b-shaped-b64-t1"])
def test_full_size_sampled_parity(built, name):
    from block_diffusion_drafter_concat_gb300.runner import StepRunner
    w = configs.BY_NAME[name]
    bs = sampled(w)
    W = orun.host_weights(w)
    seqs = {b: orun.draft_sequence(w, W, b) for b in bs}
    drafts = inputs.decoy_drafts(w).clone()
    for b in bs:
        drafts[b] = torch.as_tensor(seqs[b]["draft"])
    r = StepRunner(w)
    r.plant(drafts)
    r.step()
    torch.cuda.synchronize()
    assert r.drafter.device_error() == 0
    t, S = tol(w), w.block_size
    hid = r.hidden.view(w.batch, S, -1)
    fused = r.fused.view(w.batch, S, -1)
    rng = np.random.default_rng(0)
    checked = 0
    for b in bs:
        s = seqs[b]
        T = s["T"]
        errs = {"fused": rel_err(fused[b], s["fused"][T - S:T]), "h": rel_err(hid[b], s["h"])}
        pos = np.concatenate([np.arange(T - S, T), rng.choice(T - S, 48, replace=False)])
        for l in range(w.n_layers):
            errs[f"k{l}"] = rel_err(gather_kv(r.cache.k[l], r.table_host, b, pos), s["K"][l][pos])
            errs[f"v{l}"] = rel_err(gather_kv(r.cache.v[l], r.table_host, b, pos), s["V"][l][pos])
        print(name, b, {k: f"{v:.2e}" for k, v in errs.items()})
        assert max(errs.values()) < t, errs
        d_gpu = r.draft[b].cpu().numpy()
        slack, zg = head_parity(d_gpu, hid[b], W["lm_head"], s["z"])
        low = check_drafts(d_gpu, s["draft"], s["margin"], slack)
        print(name, b, "logit slack", f"{slack.max():.3e}", "rows left out", int(low.sum()))
        lg = r.logits[b].float().cpu().numpy()
        if w.temperature > 0:
            # verification of the GPU's drafts, whose drafter distribution is the oracle's
            # LM head on the GPU's hidden state
            u = r.uniforms[b].cpu().numpy()
            checked += check_sample(r.out_tokens[b].cpu().numpy(), r.n_acc[b], r.n_emit[b],
                                    d_gpu, zg, lg, u, w.temperature)
        else:
            checked += check_greedy(r.out_tokens[b].cpu().numpy(), r.n_acc[b].cpu(),
                                    r.n_emit[b].cpu(), d_gpu, lg)
    assert checked >= 1
    del r
    torch.cuda.empty_cache()
