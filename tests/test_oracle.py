"""Pins of the fp64 oracle against facts other than itself (closed forms, brute force,
invariants, library routines, statistics).  CPU only."""
import math
from fractions import Fraction
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O

RNG = np.random.default_rng(1234)


def tiny_cfg(**kw):
    c = dict(n_layers=2, n_q_heads=4, n_kv_heads=2, head_dim=8, rope_theta=1e4,
             rms_eps=1e-6, d=16, F=24, V=50)
    c.update(kw)
    return SimpleNamespace(**c)


def tiny_weights(cfg, rng, std=0.3):
    d, F, V = cfg.d, cfg.F, cfg.V
    qw, kvw = cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim
    W = {"embed": rng.normal(0, 1, (V, d)), "lm_head": rng.normal(0, std, (V, d)),
         "g_final": 1 + rng.normal(0, 0.1, d)}
    for l in range(cfg.n_layers):
        W[f"l{l}.g_attn"] = 1 + rng.normal(0, 0.1, d)
        W[f"l{l}.w_q"] = rng.normal(0, std, (qw, d))
        W[f"l{l}.w_k"] = rng.normal(0, std, (kvw, d))
        W[f"l{l}.w_v"] = rng.normal(0, std, (kvw, d))
        W[f"l{l}.w_o"] = rng.normal(0, std, (d, qw))
        W[f"l{l}.g_mlp"] = 1 + rng.normal(0, 0.1, d)
        W[f"l{l}.w_gate"] = rng.normal(0, std, (F, d))
        W[f"l{l}.w_up"] = rng.normal(0, std, (F, d))
        W[f"l{l}.w_down"] = rng.normal(0, std, (d, F))
    return W


def ctx_kv(cfg, rng, T, positions=None):
    pos = np.arange(T) if positions is None else positions
    K, V = [], []
    for _ in range(cfg.n_layers):
        k = rng.normal(0, 1, (T, cfg.n_kv_heads, cfg.head_dim))
        K.append(O.rope(k, pos, cfg.rope_theta))
        V.append(rng.normal(0, 1, (T, cfg.n_kv_heads, cfg.head_dim)))
    return K, V


# ------------------------------------------------------------------ bf16 rounding
def test_round_bf16_matches_library_conversion_on_fp32_inputs():
    x = np.concatenate([RNG.normal(0, 1, 20000), RNG.normal(0, 1e-3, 2000),
                        RNG.normal(0, 1e4, 2000)]).astype(np.float32)
    # exact ties: low 16 bits = 0x8000 (halfway between two bf16 values)
    exps = RNG.integers(60, 190, 4000).astype(np.uint32) << np.uint32(23)
    mant = RNG.integers(0, 2 ** 23, 4000).astype(np.uint32) & np.uint32(0x7F0000)
    ties = exps | mant | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32), -ties.view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_rounds_fp64_directly_not_through_fp32():
    # 1 + 2^-8 + 2^-40 lies above the midpoint of (1, 1 + 2^-7): nearest bf16 is
    # 1 + 2^-7; rounding to fp32 first would land on the midpoint and tie to 1.
    x = 1 + 2.0 ** -8 + 2.0 ** -40
    assert O.round_bf16(np.array([x]))[0] == 1 + 2.0 ** -7
    assert O.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0       # exact tie -> even
    assert O.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6


def test_round_bf16_is_exact_nearest_by_rational_arithmetic():
    xs = RNG.normal(0, 3, 300)
    for x in xs:
        r = O.round_bf16(np.array([x]))[0]
        e = math.frexp(abs(x))[1]             # |x| in [2^(e-1), 2^e)
        ulp = Fraction(2) ** (e - 8)
        lo = (Fraction(abs(x)) // ulp) * ulp
        cands = [lo, lo + ulp]
        best = min(cands, key=lambda c: (abs(Fraction(abs(x)) - c), (c / ulp) % 2))
        assert Fraction(abs(r)) == best and (r < 0) == (x < 0)


# ------------------------------------------------------------ closed forms
def test_rms_norm_closed_form():
    out = O.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    s = math.sqrt((9 + 16) / 2)
    np.testing.assert_allclose(out, [[3 / s, 8 / s]], rtol=1e-15)
    out = O.rms_norm(np.array([[1.0, 1.0]]), np.array([1.0, 1.0]), 1.0)
    np.testing.assert_allclose(out, [[1 / math.sqrt(2), 1 / math.sqrt(2)]], rtol=1e-15)


def test_silu_closed_form():
    np.testing.assert_allclose(O.silu(np.array([0.0, 1.0, -1.0, 40.0])),
                               [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 40.0],
                               rtol=1e-15)


def test_swiglu_mlp_closed_form_on_a_1x2_input():
    # one layer, attention switched off (W_o = 0): h = RMSNorm(x0 + W_d(silu(W_g n) * W_u n))
    cfg = tiny_cfg(n_layers=1, n_q_heads=1, n_kv_heads=1, head_dim=2, d=2, F=3, V=1)
    W = {"embed": np.array([[1.0, 2.0]]), "g_final": np.array([1.0, 1.0]),
         "lm_head": np.zeros((1, 2)),
         "l0.g_attn": np.ones(2), "l0.w_q": np.ones((2, 2)), "l0.w_k": np.ones((2, 2)),
         "l0.w_v": np.ones((2, 2)), "l0.w_o": np.zeros((2, 2)),
         "l0.g_mlp": np.array([1.0, 0.5]),
         "l0.w_gate": np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]),
         "l0.w_up": np.array([[2.0, 0.0], [0.0, -1.0], [0.5, 0.5]]),
         "l0.w_down": np.array([[1.0, 0.0, 1.0], [0.0, 1.0, -1.0]])}
    K = [np.zeros((0, 1, 2))]
    h = O.draft_block(K, K, 0, [0], W, cfg, bf16=False)
    # by hand: x0 = (1, 2); rms = sqrt(2.5); n = (1, 2*0.5)/sqrt(2.5) = (a, a)
    a = 1 / math.sqrt(2.5 + cfg.rms_eps)
    sil = lambda z: z / (1 + math.exp(-z))  # noqa: E731
    act = [sil(a) * 2 * a, sil(a) * (-a), sil(2 * a) * a]
    x = [1 + act[0] + act[2], 2 + act[1] - act[2]]
    r = math.sqrt((x[0] ** 2 + x[1] ** 2) / 2 + cfg.rms_eps)
    np.testing.assert_allclose(h, [[x[0] / r, x[1] / r]], rtol=1e-13)


def test_rope_closed_form_and_pairing():
    # head_dim 2: a plain 2-D rotation by pos radians
    out = O.rope(np.array([[[1.0, 0.0]]]), np.array([0.7]), 1e4)
    np.testing.assert_allclose(out[0, 0], [math.cos(0.7), math.sin(0.7)], rtol=1e-15)
    # head_dim 4, theta 100: pair (1, 3) turns at 100^(-1/2) = 0.1 rad per position
    out = O.rope(np.array([[[0.0, 1.0, 0.0, 0.0]]]), np.array([5]), 100.0)
    np.testing.assert_allclose(out[0, 0], [0, math.cos(0.5), 0, math.sin(0.5)],
                               atol=1e-15)
    # position 0 is the identity
    x = RNG.normal(size=(3, 2, 8))
    np.testing.assert_array_equal(O.rope(x, np.zeros(3), 1e6), x)


def test_rope_scores_depend_only_on_relative_position():
    q = RNG.normal(size=(1, 1, 16))
    k = RNG.normal(size=(1, 1, 16))
    def s(pq, pk):
        return float(np.sum(O.rope(q, [pq], 1e4) * O.rope(k, [pk], 1e4)))
    for c in (1, 17, 1000):
        assert s(5, 2) == pytest.approx(s(5 + c, 2 + c), rel=1e-10)
    assert s(5, 2) != pytest.approx(s(5, 3), rel=1e-6)


# ------------------------------------------------------------------ attention
def _brute_attention(q, k, v, hkv):
    sq, hq, hd = q.shape
    out = np.zeros_like(q)
    for i in range(sq):
        for h in range(hq):
            g = h // (hq // hkv)
            sc = [sum(q[i, h, c] * k[j, g, c] for c in range(hd)) / math.sqrt(hd)
                  for j in range(k.shape[0])]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            z = sum(e)
            for c in range(hd):
                out[i, h, c] = sum(e[j] * v[j, g, c] for j in range(k.shape[0])) / z
    return out


@pytest.mark.parametrize("sq,hq,hkv,hd,tk", [(3, 4, 2, 4, 5), (1, 1, 1, 4, 7), (2, 6, 3, 2, 1)])
def test_attention_matches_explicit_softmax_loop(sq, hq, hkv, hd, tk):
    q = RNG.normal(size=(sq, hq, hd))
    k = RNG.normal(size=(tk, hkv, hd)) * 2
    v = RNG.normal(size=(tk, hkv, hd))
    np.testing.assert_allclose(O.attention(q, k, v, hkv), _brute_attention(q, k, v, hkv),
                               rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    q = RNG.normal(size=(4, 8, 16))
    k = RNG.normal(size=(9, 2, 16))
    v = RNG.normal(size=(9, 2, 16))
    out_gqa = O.attention(q, k, v, 2)
    out_mha = O.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), 8)
    np.testing.assert_allclose(out_gqa, out_mha, rtol=1e-14)


# ------------------------------------------------------------ whole drafter
@pytest.mark.parametrize("bf16", [False, True])
def test_drafter_is_invariant_to_context_order(bf16):
    cfg = tiny_cfg()
    rng = np.random.default_rng(7)
    W = tiny_weights(cfg, rng)
    T = 11
    K, V = ctx_kv(cfg, rng, T)
    ids = [3, 0, 0, 5]
    h = O.draft_block(K, V, T, ids, W, cfg, bf16)
    perm = rng.permutation(T)
    h2 = O.draft_block([k[perm] for k in K], [v[perm] for v in V], T, ids, W, cfg, bf16)
    if bf16:   # summation order may move a value across a bf16 rounding boundary
        np.testing.assert_allclose(h2, h, atol=2e-2)
    else:
        np.testing.assert_allclose(h2, h, rtol=1e-12, atol=1e-12)


def test_drafter_is_invariant_to_a_global_position_shift():
    cfg = tiny_cfg()
    rng = np.random.default_rng(8)
    W = tiny_weights(cfg, rng)
    T = 9
    fused = rng.normal(size=(T, cfg.d))

    def run(shift, gap=0):
        pos = shift + np.arange(T)
        K, V = [], []
        for l in range(cfg.n_layers):
            k, v = O.inject_kv(fused, pos, W[f"l{l}.w_k"], W[f"l{l}.w_v"], cfg.n_kv_heads,
                               cfg.rope_theta, False)
            K.append(k)
            V.append(v)
        return O.draft_block(K, V, T, [1, 2, 3], W, cfg, False, pos0=shift + T + gap)
    np.testing.assert_allclose(run(0), run(123), rtol=1e-9, atol=1e-10)
    # control: moving the block relative to its context does change the result
    assert not np.allclose(run(0), run(0, gap=5), atol=1e-6)


def test_drafter_with_zero_sublayers_is_the_normed_embedding():
    cfg = tiny_cfg()
    rng = np.random.default_rng(9)
    W = tiny_weights(cfg, rng)
    for l in range(cfg.n_layers):
        W[f"l{l}.w_o"][:] = 0
        W[f"l{l}.w_down"][:] = 0
    K, V = ctx_kv(cfg, rng, 6)
    ids = [4, 7, 7]
    h = O.draft_block(K, V, 6, ids, W, cfg, False)
    e = W["embed"][ids]
    want = e / np.sqrt((e ** 2).mean(axis=1, keepdims=True) + cfg.rms_eps) * W["g_final"]
    np.testing.assert_allclose(h, want, rtol=1e-13)


def test_drafter_with_uniform_attention_averages_all_values():
    # W_q = 0 makes every score 0: each q head outputs the plain mean of its kv head's
    # values over context + block; one layer, MLP off.
    cfg = tiny_cfg(n_layers=1)
    rng = np.random.default_rng(10)
    W = tiny_weights(cfg, rng)
    W["l0.w_q"][:] = 0
    W["l0.w_down"][:] = 0
    T = 5
    K, V = ctx_kv(cfg, rng, T)
    ids = [2, 9]
    h = O.draft_block(K, V, T, ids, W, cfg, False)
    x0 = W["embed"][ids]
    n = x0 / np.sqrt((x0 ** 2).mean(axis=1, keepdims=True) + cfg.rms_eps) * W["l0.g_attn"]
    vb = (n @ W["l0.w_v"].T).reshape(2, cfg.n_kv_heads, cfg.head_dim)
    mean_v = (V[0].sum(axis=0) + vb.sum(axis=0)) / (T + 2)        # [hkv, hd]
    group = cfg.n_q_heads // cfg.n_kv_heads
    o = np.concatenate([mean_v[h // group] for h in range(cfg.n_q_heads)])
    x = x0 + o @ W["l0.w_o"].T
    want = x / np.sqrt((x ** 2).mean(axis=1, keepdims=True) + cfg.rms_eps) * W["g_final"]
    np.testing.assert_allclose(h, want, rtol=1e-12)


def test_fusion_scale_invariance_and_identity_reduction():
    x = RNG.normal(size=(5, 12))
    w = RNG.normal(size=(6, 12))
    g = 1 + RNG.normal(0, 0.1, 6)
    a = O.fuse_features(x, w, g, 0.0, False)
    np.testing.assert_allclose(O.fuse_features(3.5 * x, w, g, 0.0, False), a, rtol=1e-13)
    # L = 1 and W_fuse = [I]: fusion is RMSNorm of the features
    xi = RNG.normal(size=(4, 6))
    np.testing.assert_allclose(O.fuse_features(xi, np.eye(6), g, 1e-6, False),
                               O.rms_norm(xi, g, 1e-6), rtol=1e-15)
    # the layer-major concatenation: W_fuse = [0 I] picks target layer 1's block
    x2 = RNG.normal(size=(4, 12))
    w2 = np.concatenate([np.zeros((6, 6)), np.eye(6)], axis=1)
    np.testing.assert_allclose(O.fuse_features(x2, w2, g, 1e-6, False),
                               O.rms_norm(x2[:, 6:], g, 1e-6), rtol=1e-15)


# ------------------------------------------------------------------ LM head argmax
def test_lm_head_argmax_against_explicit_logits_with_ties():
    h = RNG.normal(size=(3, 5))
    w = RNG.normal(size=(40, 5))
    w[17] = w[9]                      # planted exact tie at the top for row 0
    h[0] = w[9] * 10
    z = O.lm_head(h, w)
    want = []
    for r in range(3):
        zs = [sum(h[r, c] * w[v, c] for c in range(5)) for v in range(40)]
        m = max(zs)
        want.append(min(v for v in range(40) if abs(zs[v] - m) <= 1e-9 * abs(m)))
    assert list(O.argmax_lowest(z)) == want
    assert want[0] == 9
    assert O.top2_margin(np.array([[1.0, 5.0, 3.0]]))[0] == 2.0


# ------------------------------------------------------------------ greedy verify
def _brute_greedy(draft, logits):
    S = len(draft)
    t = [int(np.flatnonzero(row == row.max())[0]) for row in logits]
    match = np.cumprod([int(draft[i] == t[i]) for i in range(S)])
    n = int(match.sum())
    return [t[i] if i <= min(n, S - 1) else -1 for i in range(S)], n, min(n + 1, S)


def test_greedy_verify_invariants_and_brute_force():
    rng = np.random.default_rng(3)
    S, V = 6, 5
    for _ in range(500):
        logits = rng.integers(0, 4, (S, V)).astype(np.float64)   # many ties
        draft = rng.integers(0, V, S)
        out, n, ne = O.verify_greedy(draft, logits)
        bo, bn, bne = _brute_greedy(draft, logits)
        assert list(out) == bo and n == bn and ne == bne
        assert 1 <= ne <= S and n <= S
    logits = rng.normal(size=(S, V))
    t = O.argmax_lowest(logits)
    out, n, ne = O.verify_greedy(t, logits)          # draft == target argmax
    assert n == S and ne == S and list(out) == list(t)
    bad = t.copy()
    bad[0] = (t[0] + 1) % V                          # mismatch at the first position
    out, n, ne = O.verify_greedy(bad, logits)
    assert n == 0 and ne == 1 and out[0] == t[0] and all(out[1:] == -1)


def test_planted_agreement_gives_the_closed_form_mean_emitted():
    from workload import synth
    S, V, p, trials = 16, 64, 0.8, 3000
    rng = np.random.default_rng(5)
    u = synth.uniform(77, "plant", (trials, S)).numpy()
    tot = 0
    for t in range(trials):
        logits = rng.normal(size=(S, V))
        draft = rng.integers(0, V, S)
        for i in range(S):
            if u[t, i] < p:
                logits[i, draft[i]] = logits[i].max() + 1.0
        tot += O.verify_greedy(draft, logits)[2]
    pe = p + (1 - p) / V             # chance agreement on unplanted positions
    want = (1 - pe ** S) / (1 - pe)
    assert abs(tot / trials - want) < 0.08


# ------------------------------------------------------------ temperature-1 verify
def _first_token_distribution(draft, zd, zt, q_mode, grid=600):
    """Probability of each first emitted token, integrating the oracle's decision over
    u[0,0] and u[0,1] on a midpoint grid."""
    V = zt.shape[1]
    prob = np.zeros(V)
    us = (np.arange(grid) + 0.5) / grid
    for a in us:
        u = np.zeros((1, 2))
        u[0, 0] = a
        out, n, _ = O.verify_sample(draft[:1], zd[:1], zt[:1], u, 1.0, q_mode)
        if n >= 1:
            prob[out[0]] += 1.0 / grid
            continue
        for b in us:
            u[0, 1] = b
            out, _, _ = O.verify_sample(draft[:1], zd[:1], zt[:1], u, 1.0, q_mode)
            prob[out[0]] += 1.0 / grid ** 2
    return prob


def test_point_mass_verify_first_token_marginal_is_the_target_distribution():
    rng = np.random.default_rng(11)
    V = 6
    zt = rng.normal(size=(1, V))
    zd = rng.normal(size=(1, V))
    draft = np.array([int(np.argmax(zd[0]))])
    p = O.softmax(zt[0])
    prob = _first_token_distribution(draft, zd, zt, "point_mass", grid=400)
    np.testing.assert_allclose(prob, p, atol=4e-3)


def test_softmax_verify_first_token_marginal_closed_form():
    rng = np.random.default_rng(12)
    V = 6
    zt = rng.normal(size=(1, V))
    zd = rng.normal(size=(1, V)) * 2
    d = int(np.argmax(zd[0]))
    p, q = O.softmax(zt[0]), O.softmax(zd[0])
    acc = min(1.0, p[d] / q[d])
    r = np.maximum(0, p - q)
    want = (1 - acc) * r / r.sum()
    want[d] += acc
    prob = _first_token_distribution(np.array([d]), zd, zt, "softmax", grid=400)
    np.testing.assert_allclose(prob, want, atol=4e-3)


def test_sample_verify_accepts_everything_when_draft_equals_target():
    rng = np.random.default_rng(13)
    S, V = 8, 30
    z = rng.normal(size=(S, V))
    d = O.argmax_lowest(z)
    u = rng.random((S, 2))
    out, n, ne = O.verify_sample(d, z, z, u, 1.0)
    assert n == S and ne == S and list(out) == list(d)


def test_sample_verify_monte_carlo_acceptance_and_residual_chi2():
    rng = np.random.default_rng(14)
    V, N = 8, 20000
    zt = rng.normal(size=(1, V))
    zd = rng.normal(size=(1, V)) * 1.5
    d = int(np.argmax(zd[0]))
    p, q = O.softmax(zt[0]), O.softmax(zd[0])
    acc_rate = min(1.0, p[d] / q[d])
    r = np.maximum(0, p - q)
    r = r / r.sum()
    n_acc, counts = 0, np.zeros(V)
    for _ in range(N):
        out, n, _ = O.verify_sample(np.array([d]), zd, zt, rng.random((1, 2)), 1.0)
        if n == 1:
            n_acc += 1
        else:
            counts[out[0]] += 1
    assert abs(n_acc / N - acc_rate) < 4 * math.sqrt(acc_rate * (1 - acc_rate) / N) + 1e-9
    rej = counts.sum()
    nz = r > 0
    chi2 = float((((counts[nz] - rej * r[nz]) ** 2) / (rej * r[nz])).sum())
    assert counts[~nz].sum() == 0
    assert chi2 < 30.0      # dof <= 7; p-value ~1e-4 at this bound
