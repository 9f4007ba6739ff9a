"""Helpers shared by the GPU parity tests (comparison rules and cache gathering)."""
import numpy as np
import torch

from oracle import dflash_oracle as O

MARGIN = 1e-2   # drafts are compared where the oracle's top-2 logit margin is >= this


def tol(w):
    return 2e-2 if w.dtype == "bf16" else 1e-4


def rel_err(gpu, ref):
    """Normwise relative error max|gpu - ref| / max|ref|."""
    g = gpu.detach().float().cpu().numpy().astype(np.float64) if torch.is_tensor(gpu) else gpu
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-30))


def gather_kv(pool, table_host, b, positions):
    """Cache rows of sequence b at `positions`: [n, n_kv_heads, head_dim] (host fp64)."""
    p = torch.as_tensor(positions, dtype=torch.int64)
    pages = table_host[b].to(torch.int64)[p // 16].to(pool.device)
    off = (p % 16).to(pool.device)
    return pool[pages, :, off, :].float().cpu().numpy().astype(np.float64)


def check_drafts(gpu_draft, oracle_draft, margin):
    """Bit-exact where the oracle's margin is >= MARGIN.  Returns the low-margin mask."""
    gpu_draft = np.asarray(gpu_draft)
    low = np.asarray(margin) < MARGIN
    bad = (~low) & (gpu_draft != np.asarray(oracle_draft))
    assert not bad.any(), (np.nonzero(bad), gpu_draft[bad], np.asarray(oracle_draft)[bad],
                           np.asarray(margin)[bad])
    return low


def check_greedy(gpu_out, gpu_nacc, gpu_nemit, draft_o, logits_row, low):
    """Greedy verify outputs of one sequence against the oracle on the oracle's drafts;
    skipped (returns False) when a low-margin draft lies at or before the oracle's
    first mismatch, since the two sides may then legitimately verify different drafts."""
    out, n, ne = O.verify_greedy(draft_o, logits_row)
    if low[: min(n, len(draft_o) - 1) + 1].any():
        return False
    assert int(gpu_nacc) == n and int(gpu_nemit) == ne, (int(gpu_nacc), n, int(gpu_nemit), ne)
    assert list(np.asarray(gpu_out)) == list(out)
    return True


def sample_ambiguous(draft, z, logits, u, tau, eps=1e-3):
    """True when a fp32 evaluation could take a different branch than fp64: an
    acceptance ratio or a residual CDF step within eps of the uniform."""
    S = len(draft)
    for i in range(S):
        p = O.softmax(logits[i] / tau)
        q = O.softmax(z[i] / tau)
        d = int(draft[i])
        if abs(u[i, 0] * q[d] - p[d]) <= eps * max(p[d], q[d]):
            return True
        if u[i, 0] < p[d] / q[d]:
            continue
        r = np.maximum(0, p - q)
        if r.sum() == 0:
            r = p
        cdf = np.cumsum(r)
        return bool(np.min(np.abs(cdf - u[i, 1] * r.sum())) <= eps * r.sum())
    return False
