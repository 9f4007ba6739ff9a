"""Plain fp64 CPU oracle of one DFlash draft + verify step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It shares no
code with the CUDA library (numpy only, no torch) and is written for a reader to check
against the pages by eye: no blocking, fusion or reordering beyond the definitions.

Pages followed (cited by title and section):
* [DFlash wiki] aisparkup.com/wiki/dflash -- "DFlash의 핵심 아이디어": block diffusion
  drafts a whole block in one parallel forward pass; "타깃 모델 피처 컨디셔닝" items
  1-3: hidden features of several target layers fused by a light projection (1),
  injected into the KV cache of every drafter layer (2), the block predicted from that
  context in one shot (3); the drafter reuses the target's embedding and LM head.
* [DFlash FAQ] opensource-hub.com/ko/library/z-lab-dflash -- FAQ 1: the target
  context goes straight into the K/V cache (KV injection) rather than into the input.
* [NVIDIA blog] "Boost inference performance up to 15x on NVIDIA Blackwell using DFlash
  speculative decoding" -- section "How does DFlash speculative decoding work?": the
  target verifies the drafted block in parallel and accepts the longest valid prefix;
  the drafter predicts a block of masked future tokens in one forward pass; target
  context features are injected into the key-value projections across the layers.

Readings where the pages are silent (each also listed in the design notes):
* fusion = one bias-free linear map of the concatenated features, then RMSNorm;
* injected K/V use each drafter layer's own W_k / W_v, RoPE at the absolute context
  position; the block's own K/V live only for this step;
* block attention is bidirectional over [context K/V of the sequence ; block K/V],
  scale 1/sqrt(head_dim), grouped-query heads (q head h uses kv head h // (hq/hkv));
* RoPE rotates the pairs (j, j + head_dim/2) by pos * theta^(-2j/head_dim);
* every argmax takes the lowest index among equal maxima;
* bf16 workloads round to bf16 (round to nearest, ties to even) at exactly these
  points: fused features; injected K/V after RoPE; each RMSNorm output that feeds a
  projection; q, k, v after RoPE; the attention output; the SwiGLU product; the final
  hidden state.  The residual stream, accumulations and softmax stay in fp64 here.

Pins (tests/test_oracle.py): bf16 rounding against the library conversion; RMSNorm,
SiLU and SwiGLU closed forms; RoPE closed form, relative-position and shift
properties; attention against an explicit per-query/per-key loop and GQA against MHA
with duplicated heads; context-permutation and position-shift invariance of the whole
drafter; the zero-sublayer and constant-value special cases of the drafter; LM-head
argmax against numpy argmax with planted ties; greedy-verify invariants and brute
force; temperature-1 verify acceptance/residual statistics and exact first-token
marginals by integration over the uniforms.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------- rounding
def round_bf16(x):
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64.

    bf16 keeps 8 significant bits; fp64 keeps 53, so the 45 low mantissa bits are
    rounded away directly from fp64 (no intermediate fp32 rounding).  Exact for zero
    and for magnitudes in the bf16 normal range (>= 2^-126), the only ones that occur
    in this computation."""
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.uint64).copy()
    keep = np.uint64(45)
    lsb = (bits >> keep) & np.uint64(1)
    bits = bits + (np.uint64((1 << 44) - 1) + lsb)
    bits &= ~np.uint64((1 << 45) - 1)
    return bits.view(np.float64)


def _maybe_bf16(x, bf16):
    return round_bf16(x) if bf16 else np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------- building blocks
def rms_norm(u, g, eps):
    """u / sqrt(mean(u^2) + eps) * g over the last axis."""
    u = np.asarray(u, dtype=np.float64)
    return u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + eps) * g


def silu(z):
    return z / (1.0 + np.exp(-z))


def rope(x, pos, theta):
    """Rotary position embedding on x [n, heads, head_dim] at positions pos [n].

    Pair (j, j + head_dim/2) is rotated by the angle pos * theta^(-2j/head_dim)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [n, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(q, k, v, n_kv_heads):
    """softmax(q k^T / sqrt(head_dim)) v with no mask, per q head.

    q [Sq, hq, hd]; k, v [Tk, hkv, hd]; q head h reads kv head h // (hq // hkv)."""
    sq, hq, hd = q.shape
    group = hq // n_kv_heads
    out = np.zeros((sq, hq, hd))
    for h in range(hq):
        g = h // group
        scores = q[:, h, :] @ k[:, g, :].T / np.sqrt(hd)          # [Sq, Tk]
        scores = scores - scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


# ------------------------------------------------------------------------- the method
def fuse_features(x_cat, w_fuse, g_fuse, eps, bf16):
    """[DFlash wiki, 타깃 모델 피처 컨디셔닝 item 1] light projection of the
    concatenated multi-layer target features: RMSNorm(X_cat W_fuse^T) * g_fuse."""
    u = np.asarray(x_cat, dtype=np.float64) @ np.asarray(w_fuse, dtype=np.float64).T
    return _maybe_bf16(rms_norm(u, g_fuse, eps), bf16)


def inject_kv(fused, positions, w_k, w_v, n_kv_heads, theta, bf16):
    """[DFlash wiki item 2; DFlash FAQ 1; NVIDIA blog, how it works] the fused
    features enter one drafter layer's cache through that layer's K/V projections:
    K = RoPE(fused W_k^T, pos), V = fused W_v^T, each [n, hkv, hd]."""
    n = fused.shape[0]
    k = (fused @ np.asarray(w_k, dtype=np.float64).T).reshape(n, n_kv_heads, -1)
    v = (fused @ np.asarray(w_v, dtype=np.float64).T).reshape(n, n_kv_heads, -1)
    return _maybe_bf16(rope(k, positions, theta), bf16), _maybe_bf16(v, bf16)


def draft_block(ctx_k, ctx_v, ctx_len, block_ids, W, cfg, bf16, trace=None, pos0=None):
    """[DFlash wiki, 블록 확산으로 병렬 드래프팅 and item 3; NVIDIA blog, how it
    works] one parallel forward pass over a block of S masked tokens at positions
    pos0 .. pos0+S-1 (pos0 = ctx_len unless given), each layer attending bidirectionally over its injected
    context K/V (ctx_k[l], ctx_v[l]: [ctx_len, hkv, hd]) and the block's own K/V, then
    a SwiGLU MLP; returns the final hidden state h [S, d] (input of the shared LM head).

    W: dict of fp64 weights named as in the workload ("l{l}.w_q", "embed", ...).
    cfg: object with n_layers, n_q_heads, n_kv_heads, head_dim, rope_theta, rms_eps.
    """
    eps, theta = cfg.rms_eps, cfg.rope_theta
    hq, hkv = cfg.n_q_heads, cfg.n_kv_heads
    S = len(block_ids)
    pos = (ctx_len if pos0 is None else pos0) + np.arange(S)
    x = np.asarray(W["embed"], dtype=np.float64)[np.asarray(block_ids)]   # [S, d]
    for l in range(cfg.n_layers):
        L = lambda name: W[f"l{l}.{name}"]  # noqa: E731
        n = _maybe_bf16(rms_norm(x, L("g_attn"), eps), bf16)
        q = rope((n @ L("w_q").T).reshape(S, hq, -1), pos, theta)
        k = rope((n @ L("w_k").T).reshape(S, hkv, -1), pos, theta)
        v = (n @ L("w_v").T).reshape(S, hkv, -1)
        q, k, v = (_maybe_bf16(t, bf16) for t in (q, k, v))
        keys = np.concatenate([ctx_k[l][:ctx_len], k], axis=0)
        vals = np.concatenate([ctx_v[l][:ctx_len], v], axis=0)
        o = _maybe_bf16(attention(q, keys, vals, hkv).reshape(S, -1), bf16)
        x = x + o @ L("w_o").T
        n2 = _maybe_bf16(rms_norm(x, L("g_mlp"), eps), bf16)
        act = _maybe_bf16(silu(n2 @ L("w_gate").T) * (n2 @ L("w_up").T), bf16)
        x = x + act @ L("w_down").T
        if trace is not None:
            trace.append(dict(q=q, k=k, v=v, o=o, x=x.copy()))
    return _maybe_bf16(rms_norm(x, W["g_final"], eps), bf16)


def lm_head(h, w_lm):
    """[DFlash wiki: the drafter reuses the target's LM head] logits z = h W_lm^T."""
    return np.asarray(h, dtype=np.float64) @ np.asarray(w_lm, dtype=np.float64).T


def argmax_lowest(z):
    """Index of the largest value of each row, lowest index among equal maxima."""
    return np.argmax(np.asarray(z), axis=-1)


def top2_margin(z):
    """Largest minus second-largest value of each row."""
    part = np.partition(np.asarray(z, dtype=np.float64), -2, axis=-1)
    return part[..., -1] - part[..., -2]


def verify_greedy(draft, target_logits):
    """[NVIDIA blog, how it works: accept the longest valid prefix] greedy verify of
    one sequence.  t_i = argmax of target row i; n = number of leading i with
    draft_i == t_i; emitted tokens are t_0 .. t_min(n, S-1) (the accepted drafts plus
    one target token when n < S).

    Returns (out_tokens [S] padded with -1, n_accepted, n_emitted)."""
    draft = np.asarray(draft)
    S = len(draft)
    t = argmax_lowest(target_logits)
    n = 0
    while n < S and draft[n] == t[n]:
        n += 1
    n_emit = min(n + 1, S)
    out = np.full(S, -1, dtype=np.int64)
    out[:n_emit] = t[:n_emit]
    return out, n, n_emit


def softmax(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def verify_sample(draft, draft_logits, target_logits, u, temperature=1.0,
                  q_mode="softmax"):
    """Temperature-tau verify of one sequence with supplied uniforms u [S, 2].

    p_i = softmax(target_i / tau); q_i = softmax(z_i / tau) (q_mode "softmax") or the
    point mass on draft_i (q_mode "point_mass").  Walking i = 0..S-1, draft_i is
    accepted iff u[i,0] < p_i(d_i) / q_i(d_i).  At the first rejection n the emitted
    token is drawn from r = max(0, p_n - q_n) (r = p_n when that is all zero) by
    inverse CDF: the lowest v with sum_{w<=v} r_w >= u[n,1] * sum(r), else the last v
    with r_v > 0.  Returns (out_tokens [S] padded with -1, n_accepted, n_emitted)."""
    draft = np.asarray(draft)
    S, V = np.asarray(target_logits).shape
    out = np.full(S, -1, dtype=np.int64)
    for i in range(S):
        p = softmax(np.asarray(target_logits[i], dtype=np.float64) / temperature)
        if q_mode == "softmax":
            q = softmax(np.asarray(draft_logits[i], dtype=np.float64) / temperature)
        else:
            q = np.zeros(V)
            q[draft[i]] = 1.0
        d = int(draft[i])
        if u[i, 0] < p[d] / q[d]:
            out[i] = d
            continue
        r = np.maximum(0.0, p - q)
        if r.sum() == 0.0:
            r = p
        Z = r.sum()
        cdf = np.cumsum(r)
        hit = np.nonzero(cdf >= u[i, 1] * Z)[0]
        out[i] = int(hit[0]) if len(hit) else int(np.nonzero(r > 0)[0][-1])
        return out, i, i + 1
    return out, S, S


# --------------------------------------------------------------- one sequence, one step
def draft_step(x_cat, ctx_len, block_ids, W, cfg, bf16):
    """Fuse + inject the context features of one sequence (positions 0..ctx_len-1),
    then draft the block at positions ctx_len.. and take the LM-head argmax.

    Returns dict(fused, K, V (lists per layer), h, z, draft, margin)."""
    fused = fuse_features(x_cat[:ctx_len], W["w_fuse"], W["g_fuse"], cfg.rms_eps, bf16)
    pos = np.arange(ctx_len)
    K, V = [], []
    for l in range(cfg.n_layers):
        k, v = inject_kv(fused, pos, W[f"l{l}.w_k"], W[f"l{l}.w_v"], cfg.n_kv_heads,
                         cfg.rope_theta, bf16)
        K.append(k)
        V.append(v)
    h = draft_block(K, V, ctx_len, block_ids, W, cfg, bf16)
    z = lm_head(h, W["lm_head"])
    return dict(fused=fused, K=K, V=V, h=h, z=z, draft=argmax_lowest(z),
                margin=top2_margin(z))


# ------------------------------------------------ causal passes (input fusion, target)
def causal_attention(q, k, v, n_kv_heads, n_prefix):
    """softmax(q k^T / sqrt(head_dim)) v for Sq new tokens after n_prefix cached ones:
    new token i sees the n_prefix cached keys and the new keys 0..i.

    q [Sq, hq, hd]; k, v [n_prefix + Sq, hkv, hd]; q head h reads kv head h // (hq // hkv)."""
    sq, hq, hd = q.shape
    group = hq // n_kv_heads
    seen = np.arange(n_prefix + sq)[None, :] <= n_prefix + np.arange(sq)[:, None]   # [Sq, Tk]
    out = np.zeros((sq, hq, hd))
    for h in range(hq):
        g = h // group
        scores = q[:, h, :] @ k[:, g, :].T / np.sqrt(hd)
        scores = np.where(seen, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        p = np.exp(scores)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ v[:, g, :]
    return out


def causal_stack(x, W, cfg, bf16, tap_layers=()):
    """The layer stack run causally over a whole sequence of N tokens at positions
    0..N-1 whose layer-0 inputs are the rows of x [N, d] (a token embedding, or fused
    target features in the input-fusion variant): per layer RMSNorm, Q/K/V + RoPE,
    causal attention (token i sees tokens 0..i), output projection + residual, RMSNorm,
    SwiGLU MLP + residual, with the rounding points of draft_block.

    Returns (K, V, taps, h): per-layer K/V [N, hkv, hd] (what a cache holds), the
    residual stream after each layer in tap_layers (1-based) concatenated [N, n*d]
    (rounded like a stored feature), and the final RMSNorm output h [N, d]."""
    eps, theta = cfg.rms_eps, cfg.rope_theta
    hq, hkv = cfg.n_q_heads, cfg.n_kv_heads
    x = np.asarray(x, dtype=np.float64)
    N = x.shape[0]
    pos = np.arange(N)
    K, V, taps = [], [], {}
    for l in range(cfg.n_layers):
        L = lambda name: W[f"l{l}.{name}"]  # noqa: E731
        n = _maybe_bf16(rms_norm(x, L("g_attn"), eps), bf16)
        q = _maybe_bf16(rope((n @ L("w_q").T).reshape(N, hq, -1), pos, theta), bf16)
        k = _maybe_bf16(rope((n @ L("w_k").T).reshape(N, hkv, -1), pos, theta), bf16)
        v = _maybe_bf16((n @ L("w_v").T).reshape(N, hkv, -1), bf16)
        K.append(k)
        V.append(v)
        o = _maybe_bf16(causal_attention(q, k, v, hkv, 0).reshape(N, -1), bf16)
        x = x + o @ L("w_o").T
        n2 = _maybe_bf16(rms_norm(x, L("g_mlp"), eps), bf16)
        act = _maybe_bf16(silu(n2 @ L("w_gate").T) * (n2 @ L("w_up").T), bf16)
        x = x + act @ L("w_down").T
        if l + 1 in tap_layers:
            taps[l + 1] = _maybe_bf16(x, bf16)
    tap = np.concatenate([taps[t] for t in tap_layers], axis=1) if tap_layers else None
    return K, V, tap, _maybe_bf16(rms_norm(x, W["g_final"], eps), bf16)


def input_fusion_context(fused, W, cfg, bf16):
    """[DFlash FAQ 1, the input-fusion ablation] the fused target features of the
    context tokens are the drafter's input: they run through the drafter's layers
    causally (full per-token processing, which KV injection skips) and each layer's
    K/V of the context tokens are what the block then attends to.  Returns (K, V)."""
    K, V, _, _ = causal_stack(fused, W, cfg, bf16)
    return K, V


def draft_step_input_fusion(x_cat, ctx_len, block_ids, W, cfg, bf16):
    """draft_step for the input-fusion variant: fuse the context features, run them
    through the layer stack (input_fusion_context), draft the block, LM head."""
    fused = fuse_features(x_cat[:ctx_len], W["w_fuse"], W["g_fuse"], cfg.rms_eps, bf16)
    K, V = input_fusion_context(fused, W, cfg, bf16)
    h = draft_block(K, V, ctx_len, block_ids, W, cfg, bf16)
    z = lm_head(h, W["lm_head"])
    return dict(fused=fused, K=K, V=V, h=h, z=z, draft=argmax_lowest(z), margin=top2_margin(z))


def target_forward(tokens, Wt, cfg_t, bf16, tap_layers):
    """A plain causal transformer (the target of the speculative loop) over tokens
    0..N-1: returns (taps [N, n_taps*d], logits [N, V]); row p of the logits scores the
    token at position p + 1."""
    x = np.asarray(Wt["embed"], dtype=np.float64)[np.asarray(tokens)]
    _, _, taps, h = causal_stack(x, Wt, cfg_t, bf16, tap_layers)
    return taps, lm_head(h, Wt["lm_head"])


def plant_agreement(logits, drafts, u, p):
    """Synthetic agreement of the loop's target with the drafter (no trained pair exists
    here): row i of the block's target logits gets logit[draft_{i+1}] = max_i + 1 when
    u_i < p (i < S-1).  Returns a planted copy."""
    out = np.array(logits, dtype=np.float64, copy=True)
    for i in range(out.shape[0] - 1):
        if u[i] < p:
            out[i, drafts[i + 1]] = out[i].max() + 1.0
    return out


def spec_step(committed, draft_fn, Wt, cfg_t, bf16, tap_layers, S, plant_u=None, plant_p=0.0):
    """[DFlash wiki, 사용법 (spec_generate); NVIDIA blog, how it works: draft a block,
    verify it with the target in one pass, accept the longest valid prefix] one step of
    greedy speculative decoding.  committed: the tokens so far (the last one is the
    anchor, not yet processed by the target).  draft_fn(committed, feats) -> drafts
    [S] for block slots 1..S-1 (slot 0 is the anchor; drafts[0] is ignored), where feats
    are the target's tap features of tokens 0..len-2.

    The target runs over [committed ; drafts 1..S-1]; its logits at the anchor and the
    drafts, t_i = argmax row i (lowest index), accept d_{i+1} while it equals t_i; the
    emitted tokens are t_0..t_n (the accepted drafts and one target token).
    Returns (emitted tokens, n accepted, drafts, the block's target logits)."""
    N = len(committed)
    feats, _ = target_forward(committed[:N - 1], Wt, cfg_t, bf16, tap_layers) if N > 1 else \
        (None, None)
    drafts = np.asarray(draft_fn(committed, feats))
    seq = np.concatenate([committed, drafts[1:S]])
    _, logits = target_forward(seq, Wt, cfg_t, bf16, tap_layers)
    block = logits[N - 1:N - 1 + S]
    if plant_u is not None:
        block = plant_agreement(block, drafts, plant_u, plant_p)
    t = argmax_lowest(block)
    n = 0
    while n < S - 1 and drafts[n + 1] == t[n]:
        n += 1
    return t[:n + 1], n, drafts, block


def greedy_decode(prompt, n_new, Wt, cfg_t, bf16):
    """Plain autoregressive greedy decoding of the target (the reference that lossless
    speculative decoding must reproduce token for token)."""
    seq = list(prompt)
    for _ in range(n_new):
        _, logits = target_forward(np.asarray(seq), Wt, cfg_t, bf16, ())
        seq.append(int(argmax_lowest(logits[-1])))
    return seq[len(prompt):]


def dflash_drafter(W, cfg, bf16, mask_id=0, variant="kv"):
    """draft_fn of spec_step for the DFlash drafter: fuse the context's target features,
    put them into every layer's K/V (variant "kv": inject_kv at positions 0..T-1;
    "input": input_fusion_context), draft the block [anchor, mask, ..., mask] at
    positions T..T+S-1, LM-head argmax.  The function also records each call's logits
    in fn.calls (for margin checks)."""
    S = cfg.block_size

    def fn(committed, feats):
        T = len(committed) - 1
        fused = fuse_features(feats, W["w_fuse"], W["g_fuse"], cfg.rms_eps, bf16)
        if variant == "kv":
            K, V = [], []
            for l in range(cfg.n_layers):
                k, v = inject_kv(fused, np.arange(T), W[f"l{l}.w_k"], W[f"l{l}.w_v"],
                                 cfg.n_kv_heads, cfg.rope_theta, bf16)
                K.append(k)
                V.append(v)
        else:
            K, V = input_fusion_context(fused, W, cfg, bf16)
        ids = np.full(S, mask_id)
        ids[0] = committed[-1]
        z = lm_head(draft_block(K, V, T, ids, W, cfg, bf16), W["lm_head"])
        fn.calls.append(z)
        return argmax_lowest(z)

    fn.calls = []
    return fn


# ------------------------------------------------------- low-precision weight streaming
E4M3_MAX = 448.0   # largest finite float8 e4m3 value: 1.75 * 2^8


def round_e4m3(x):
    """Round fp64 values to the nearest float8 e4m3 value (1 sign, 4 exponent bits with
    bias 7, 3 mantissa bits; subnormals in steps of 2^-9; no infinities), ties to even,
    for |x| <= 448.  Returned as fp64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                        # below 2^-6 the spacing stays 2^-9
    ulp = np.exp2(e - 3.0)
    return np.sign(x) * np.round(a / ulp) * ulp    # np.round: halves to even


def quantize_rows_fp8(w):
    """[NVIDIA blog, Blackwell Ultra paragraph: low-precision tensor formats] per output
    row n of an [out, in] matrix: a power-of-two scale s_n = 2^ceil(log2(max|w_n| / 448))
    (1 for an all-zero row), so that w / s is exact and at most 448 in magnitude, and
    codes q = e4m3(w / s).  Returns (q [out, in] as fp64 values, s [out])."""
    w = np.asarray(w, dtype=np.float64)
    amax = np.abs(w).max(axis=1)
    s = np.where(amax > 0, np.exp2(np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E4M3_MAX))),
                 1.0)
    return round_e4m3(w / s[:, None]), s


FP8_MATRICES = ("w_fuse", "w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "lm_head")


def fp8_weights(W):
    """The drafter's weights as the FP8 weight-streaming path holds them: every
    projection matrix (fusion, Q/K/V/O, gate/up/down, LM head) replaced by its
    dequantized per-row FP8 form q * s; embedding and gains unchanged."""
    out = dict(W)
    for name, m in W.items():
        if name.split(".")[-1] in FP8_MATRICES:
            q, s = quantize_rows_fp8(m)
            out[name] = q * s[:, None]
    return out
