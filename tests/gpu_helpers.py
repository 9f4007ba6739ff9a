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


def check_drafts(gpu_draft, oracle_draft, margin, slack=None):
    """Bit-exact where the oracle's top-2 margin is >= MARGIN and, per row, >= `slack`
    when given.  Returns the mask of rows left out."""
    gpu_draft = np.asarray(gpu_draft)
    low = np.asarray(margin) < MARGIN
    if slack is not None:
        low |= np.asarray(margin) < np.asarray(slack)
    bad = (~low) & (gpu_draft != np.asarray(oracle_draft))
    assert not bad.any(), (np.nonzero(bad), gpu_draft[bad], np.asarray(oracle_draft)[bad],
                           np.asarray(margin)[bad])
    return low


def check_greedy(gpu_out, gpu_nacc, gpu_nemit, gpu_draft, logits_row):
    """Greedy verify outputs of one sequence, bit-exact against the oracle's verification
    of the same drafts (the GPU's, which the draft checks tie to the oracle's) with the
    same target logits."""
    out, n, ne = O.verify_greedy(np.asarray(gpu_draft), logits_row)
    assert int(gpu_nacc) == n and int(gpu_nemit) == ne, (int(gpu_nacc), n, int(gpu_nemit), ne)
    assert list(np.asarray(gpu_out)) == list(out)
    return True


def check_sample(gpu_out, gpu_nacc, gpu_nemit, draft, z, logits, u, tau, eps=1e-3,
                 cdf_tol=1e-4):
    """Temperature-tau verify outputs of one sequence against the oracle's walk over the
    same drafts, drafter logits z, target logits and uniforms.

    The acceptance decisions are compared exactly; a walk that meets a ratio within eps
    of its uniform is left unchecked (returns False).  At a rejection the residual token
    is drawn by inverse CDF over the whole vocabulary: with 10^5 entries the CDF steps
    are far finer than what an fp32 sum resolves, so the unique part is compared (the
    rejection slot, the accepted prefix) and the drawn token must be a valid draw: its
    CDF interval must contain u * sum(r) to within cdf_tol * sum(r)."""
    gpu_out = np.asarray(gpu_out)
    draft = np.asarray(draft)
    S = len(draft)
    for i in range(S):
        p = O.softmax(np.asarray(logits[i], dtype=np.float64) / tau)
        q = O.softmax(np.asarray(z[i], dtype=np.float64) / tau)
        d = int(draft[i])
        if abs(u[i, 0] * q[d] - p[d]) <= eps * max(p[d], q[d]):
            return False
        if u[i, 0] < p[d] / q[d]:
            continue
        assert (int(gpu_nacc), int(gpu_nemit)) == (i, i + 1), (int(gpu_nacc), int(gpu_nemit), i)
        assert list(gpu_out[:i]) == list(draft[:i])
        r = np.maximum(0.0, p - q)
        if r.sum() == 0.0:
            r = p
        Z = r.sum()
        cdf = np.cumsum(r)
        t = int(gpu_out[i])
        assert 0 <= t < len(r) and r[t] > 0, t
        lo = cdf[t - 1] if t > 0 else 0.0
        assert lo - cdf_tol * Z <= u[i, 1] * Z <= cdf[t] + cdf_tol * Z, (t, lo, cdf[t], u[i, 1] * Z)
        return True
    assert (int(gpu_nacc), int(gpu_nemit)) == (S, S)
    assert list(gpu_out) == list(draft)
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


def head_parity(gpu_draft, h_gpu, w_lm, z_oracle=None):
    """The LM head + argmax on identical input, then the GPU's logit deviation.

    The oracle's LM head applied to the GPU's own final hidden state must pick the
    GPU's draft wherever that margin is >= MARGIN (the head adds no error of its own).
    Returns (dz, zg): dz [rows] = max_v |z(h_gpu) - z_oracle| per row (None without
    z_oracle), the logit change that the GPU's hidden-state difference causes, and zg =
    the oracle's logits of the GPU's hidden state."""
    hg = np.asarray(h_gpu.detach().float().cpu().numpy() if torch.is_tensor(h_gpu) else h_gpu,
                    dtype=np.float64)
    zg = O.lm_head(hg, w_lm)
    check_drafts(gpu_draft, O.argmax_lowest(zg), O.top2_margin(zg))
    dz = None if z_oracle is None else np.abs(zg - np.asarray(z_oracle)).max(axis=-1)
    return dz, zg


def capped_draft_check(name, gpu_draft, oracle_draft, margin, dz):
    """End-to-end draft parity with the slack capped by the oracle-derived constant of
    workload `name`: dz (the GPU's per-row logit deviation) must stay within the cap,
    and rows whose oracle margin is >= max(MARGIN, 2 dz) must match bit-exactly.
    Returns (rows checked, rows left out)."""
    from parity_plan import cap
    c = cap(name)
    dz = np.asarray(dz)
    assert dz.max() <= c, f"{name}: GPU logit deviation {dz.max():.4g} exceeds the cap {c:.4g}"
    low = check_drafts(gpu_draft, oracle_draft, margin, 2.0 * dz)
    return int((~low).sum()), int(low.sum())
