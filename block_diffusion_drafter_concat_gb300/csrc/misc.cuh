// Row kernels of the drafter step: block embedding + RMSNorm, RMSNorm, the LM-head
// argmax finalisation, and the verification kernels (greedy, temperature tau).
#pragma once

#include "common.cuh"

namespace dflash {

constexpr int kRowThreads = 256;

// Block-wide sum over kRowThreads threads (fixed tree: deterministic).
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
  return t;
}

// y[m] = x[m] / sqrt(mean(x[m]^2) + eps) * g, one CTA per row.
// With `ids`, x[m] is first set to the embedding row ids[m] (block embedding), with
// `rows` (and no ids) to rows[m] (input rows of a chunk of context), and in both cases
// the position ctx_lens[m / S] + m % S is written to pos[m] and x[m] to xout.
// With `xin2`, the CTAs m >= m2 normalise a second set of rows in the same launch:
// y[m] = xin2[m - m2] / rms * gain2 (the fused context rows that follow the block's
// rows in the first projection's input).
template <typename T, typename Tin>
__global__ void __launch_bounds__(kRowThreads)
    k_rmsnorm(const Tin* __restrict__ xin, float* __restrict__ xout, const T* __restrict__ gain,
              T* __restrict__ y, int d, float eps, const int* __restrict__ ids,
              const T* __restrict__ embed, int vocab, const int* __restrict__ ctx_lens, int S,
              int max_position, int* __restrict__ pos, int* err, const T* __restrict__ rows,
              const Tin* __restrict__ xin2, const T* __restrict__ gain2, int m2) {
  __shared__ float red[kRowThreads / 32];
  const int m = blockIdx.x;
  if (xin2 && m >= m2) {
    xin = xin2 - (long long)m2 * d;   // so that xin + m * d is row m - m2 of xin2
    gain = gain2;
    ids = nullptr;
    rows = nullptr;
  }
  // the gains are weights (never written on the device): fetch them before the wait
  float gv[32];
  const bool regs = (sizeof(Tin) == 4) && (d & 3) == 0 && d <= kRowThreads * 4 * 8 && !ids &&
                    !rows;
  if (regs) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = (k * kRowThreads + threadIdx.x) * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) gv[k * 4 + q] = c + q < d ? to_f32<T>(gain[c + q]) : 0.f;
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  const Tin* src = xin + (long long)m * d;
  if (ids || rows) {
    int id = ids ? ids[m] : 0;
    const int b = m / S, i = m % S;
    const int p = ctx_lens[b] + i;
    if (threadIdx.x == 0) {
      pos[m] = p;
      if (p < 0 || p >= max_position || ctx_lens[b] < 0) raise_error(err, DFLASH_DEV_BAD_POSITION);
    }
    if (ids && (id < 0 || id >= vocab)) {
      if (threadIdx.x == 0) raise_error(err, DFLASH_DEV_BAD_INDEX);
      id = 0;
    }
    src = nullptr;
    const T* e = ids ? embed + (long long)id * d : rows + (long long)m * d;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d; c += kRowThreads) {
      float v = to_f32<T>(e[c]);
      xout[(long long)m * d + c] = v;
      ss += v * v;
    }
    const float rs = 1.0f / sqrtf(block_sum(ss, red) / d + eps);
    for (int c = threadIdx.x; c < d; c += kRowThreads)
      y[(long long)m * d + c] = from_f32<T>(to_f32<T>(e[c]) * rs * to_f32<T>(gain[c]));
    return;
  }
  if constexpr (sizeof(Tin) == 4) {
    if (regs) {
      // the row stays in registers: up to 8 float4 per thread, all loads in flight
      float4 v[8];
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = (k * kRowThreads + threadIdx.x) * 4;
        if (c < d) {
          v[k] = *reinterpret_cast<const float4*>(src + c);
          ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        }
      }
      const float rs = 1.0f / sqrtf(block_sum(ss, red) / d + eps);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = (k * kRowThreads + threadIdx.x) * 4;
        if (c < d) {
          T* o = y + (long long)m * d + c;
          o[0] = from_f32<T>(v[k].x * rs * gv[k * 4]);
          o[1] = from_f32<T>(v[k].y * rs * gv[k * 4 + 1]);
          o[2] = from_f32<T>(v[k].z * rs * gv[k * 4 + 2]);
          o[3] = from_f32<T>(v[k].w * rs * gv[k * 4 + 3]);
        }
      }
      return;
    }
  }
  float ss = 0.f;
  for (int c = threadIdx.x; c < d; c += kRowThreads) {
    float v = to_f32<Tin>(src[c]);
    ss += v * v;
  }
  const float rs = 1.0f / sqrtf(block_sum(ss, red) / d + eps);
  for (int c = threadIdx.x; c < d; c += kRowThreads)
    y[(long long)m * d + c] = from_f32<T>(to_f32<Tin>(src[c]) * rs * to_f32<T>(gain[c]));
}

// Reduce the LM head's per-tile (max, argmax, sum exp) partials of each row in tile
// order: tokens = argmax (lowest index), max_logit, lse = max/tau + log(sum).
static __global__ void __launch_bounds__(kRowThreads)
    k_argmax_finalize(const float* __restrict__ am_max, const int* __restrict__ am_idx,
                      const float* __restrict__ am_sum, int n_tiles, int M, float inv_temp,
                      int* __restrict__ tokens, float* __restrict__ max_logit,
                      float* __restrict__ lse) {
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * (kRowThreads / 32) + warp;
  if (m >= M) return;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int t = lane; t < n_tiles; t += 32) {
    float v = am_max[(long long)t * M + m];
    int i = am_idx[(long long)t * M + m];
    if (v > best || (v == best && i < bi)) { best = v; bi = i; }
  }
  warp_argmax(best, bi);
  if (lane == 0) tokens[m] = bi;
  if (lse) {
    // each lane sums its tiles rescaled to the row maximum, lanes in a fixed tree
    float s = 0.f;
    for (int t = lane; t < n_tiles; t += 32)
      s += am_sum[(long long)t * M + m] * __expf((am_max[(long long)t * M + m] - best) * inv_temp);
    s = warp_sum(s);
    if (lane == 0) lse[m] = best * inv_temp + logf(s);
  }
  if (max_logit && lane == 0) max_logit[m] = best;
}

// ------------------------------------------------------- chunk K/V into the cache
// The K/V of a causal chunk (S rows per sequence, in the attention layout
// [B][hkv][S][hd]) are written into the layer's cache pages at positions
// ctx_lens[b] + i: page page_table[b][p / 16], offset p % 16.  grid (B*S), one CTA per
// row; threads walk the row's hkv*hd K and V elements 16 bytes at a time.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    k_chunk_kv_to_cache(const T* __restrict__ kb, const T* __restrict__ vb,
                        const int* __restrict__ ctx_lens, const int* __restrict__ page_table,
                        int max_pages, int num_pages, T* __restrict__ kpool,
                        T* __restrict__ vpool, int S, int hkv, int hd, int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x, b = m / S, i = m % S;
  const int p = ctx_lens[b] + i;
  const int pi = p / kPage;
  if (p < 0 || pi >= max_pages) {
    if (threadIdx.x == 0) raise_error(err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  const int page = page_table[(long long)b * max_pages + pi];
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) raise_error(err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  constexpr int VEC = 16 / sizeof(T);
  const int per_head = hd / VEC;
  for (int x = threadIdx.x; x < 2 * hkv * per_head; x += kRowThreads) {
    const int kv = x / (hkv * per_head), rem = x % (hkv * per_head);
    const int g = rem / per_head, c = (rem % per_head) * VEC;
    const T* src = (kv ? vb : kb) + (((long long)b * hkv + g) * S + i) * hd + c;
    T* dst = (kv ? vpool : kpool) + (((long long)page * hkv + g) * kPage + p % kPage) * hd + c;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// ------------------------------------------------------------------ FP8 packing
// One CTA per row of a bf16 [rows, cols] matrix: the smallest e with max|w| <= 448 * 2^e
// (exact fp32 comparisons with powers of two), scale 2^e, codes e4m3(w * 2^-e) rounded
// to nearest even (w * 2^-e is exact), zero codes in the row's padding up to ld.
static __global__ void __launch_bounds__(kRowThreads)
    k_pack_fp8(const bf16* __restrict__ w, int cols, uint8_t* __restrict__ codes, int ld,
               float* __restrict__ scales) {
  __shared__ float red[kRowThreads / 32];
  __shared__ int se;
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const bf16* row = w + (long long)r * cols;
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += kRowThreads) amax = fmaxf(amax, fabsf(to_f32<bf16>(row[c])));
  amax = warp_max(amax);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = red[0];
    for (int k = 1; k < kRowThreads / 32; ++k) a = fmaxf(a, red[k]);
    int e = 0;
    if (a > 0.f) {
      e = ilogbf(a) - 8;                            // 448 = 1.75 * 2^8
      while (a > ldexpf(448.f, e)) ++e;
      while (a <= ldexpf(448.f, e - 1)) --e;
    }
    se = e;
    scales[r] = ldexpf(1.f, e);
  }
  __syncthreads();
  const int e = se;
  uint8_t* out = codes + (long long)r * ld;
  for (int c = threadIdx.x; c < ld; c += kRowThreads)
    out[c] = c < cols ? static_cast<uint8_t>(__nv_cvt_float_to_fp8(ldexpf(to_f32<bf16>(row[c]), -e),
                                                                    __NV_SATFINITE, __NV_E4M3))
                      : 0;
}

// ------------------------------------------------------------------ layer taps
// out[m, col0 + c] = x[m, c] (fp32 residual stream -> storage dtype) for c < d: the
// hidden state after one layer, stored as one column block of a feature row.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    k_tap(const float* __restrict__ x, int d, T* __restrict__ out, int ld_out, int col0) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x;
  for (int c = threadIdx.x; c < d; c += kRowThreads)
    out[(long long)m * ld_out + col0 + c] = from_f32<T>(x[(long long)m * d + c]);
}

// ------------------------------------------------------------------ greedy verify
// grid (chunks, B*S).  Each CTA takes the argmax (lowest index) of one vocab chunk of
// one target row; the last CTA of a sequence reduces the chunks, walks the block and
// writes the accepted prefix plus the bonus token.  `shift` = 0: row i verifies draft
// slot i (every slot drafted); 1: row i verifies slot i + 1 (slot 0 holds the anchor
// token, whose target row scores the first draft), so at most S - 1 are accepted.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    k_verify_greedy(const T* __restrict__ logits, const int* __restrict__ draft, int S, int V,
                    int chunk, float* __restrict__ part_v, int* __restrict__ part_i,
                    int* __restrict__ counters, int* __restrict__ out_tokens,
                    int* __restrict__ n_acc, int* __restrict__ n_emit, int* err,
                    int shift) {
  __shared__ float sv[kRowThreads / 32];
  __shared__ int si[kRowThreads / 32];
  __shared__ int flag;
  __shared__ int tok[64];
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int b = row / S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* src = logits + (long long)row * V;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  float best = -INFINITY;
  int bi = 0x7fffffff;
  constexpr int VEC = 16 / sizeof(T);
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(src + v0) & 15) == 0);
  if (vec_ok) {
    const int nv = (v1 - v0) / VEC;
    for (int k = threadIdx.x; k < nv; k += kRowThreads) {
      uint4 raw = __ldcs(reinterpret_cast<const uint4*>(src + v0) + k);
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        float v = to_f32<T>(e[j]);
        if (v > best) { best = v; bi = v0 + k * VEC + j; }
      }
    }
    for (int v = v0 + nv * VEC + threadIdx.x; v < v1; v += kRowThreads) {
      float x = to_f32<T>(src[v]);
      if (x > best) { best = x; bi = v; }
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += kRowThreads) {
      float x = to_f32<T>(src[v]);
      if (x > best) { best = x; bi = v; }
    }
  }
  warp_argmax(best, bi);
  if (lane == 0) { sv[warp] = best; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kRowThreads / 32; ++w)
      if (sv[w] > best || (sv[w] == best && si[w] < bi)) { best = sv[w]; bi = si[w]; }
    part_v[(long long)row * nch + c] = best;
    part_i[(long long)row * nch + c] = bi;
  }
  if (!elect_last(&counters[b], S * nch, &flag)) return;
  // last CTA of sequence b: one warp per block slot
  for (int i = warp; i < S; i += kRowThreads / 32) {
    float bv = -INFINITY;
    int bx = 0x7fffffff;
    const long long r = (long long)b * S + i;
    for (int k = lane; k < nch; k += 32) {
      float v = __ldcg(part_v + r * nch + k);
      int x = __ldcg(part_i + r * nch + k);
      if (v > bv || (v == bv && x < bx)) { bv = v; bx = x; }
    }
    warp_argmax(bv, bx);
    if (lane == 0) tok[i] = bx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = 0;
    while (n < S - shift) {
      int dft = draft[(long long)b * S + shift + n];
      if (dft < 0 || dft >= V) { raise_error(err, DFLASH_DEV_BAD_INDEX); break; }
      if (dft != tok[n]) break;
      ++n;
    }
    const int ne = min(n + 1, S);
    for (int i = 0; i < S; ++i) out_tokens[(long long)b * S + i] = i < ne ? tok[i] : -1;
    n_acc[b] = n;
    n_emit[b] = ne;
  }
}

// ------------------------------------------------------------ temperature-tau verify
// Eight consecutive values as floats from a 16-byte aligned address.
__device__ __forceinline__ void load8_stream(const bf16* p, float (&x)[8]) {
  const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(p));
  const bf16* e = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = __bfloat162float(e[j]);
}
__device__ __forceinline__ void load8_stream(const float* p, float (&x)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const bf16* p, float (&x)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const bf16* e = reinterpret_cast<const bf16*>(&raw);
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = __bfloat162float(e[j]);
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *(reinterpret_cast<const float4*>(p) + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Merges running (max m, sum s of exp((x - m) * it)) states.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2, float it) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
  } else if (m2 > m) {
    s = s * __expf((m - m2) * it) + s2;
    m = m2;
  } else {
    s += s2 * __expf((m2 - m) * it);
  }
}

// Pass 1, grid (chunks, B*S): per chunk of target row r the max and sum exp of
// logits/tau; the last CTA of a row forms lse_t[r] and p_r(d_r); the last row of a
// sequence walks the acceptance test u[i,0] < p_i(d_i) / q_i(d_i), writes the accepted
// prefix, and records the first rejected slot (or S) in rej[b]; it also copies that
// slot's hidden row into hrow[b] for the drafter-logit recompute.
template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    k_verify_sample_accept(const T* __restrict__ logits, const int* __restrict__ draft,
                           const float* __restrict__ dmax, const float* __restrict__ dlse,
                           const float* __restrict__ u, const T* __restrict__ hidden, int d,
                           int S, int V, int chunk, float inv_temp,
                           float* __restrict__ part_m, float* __restrict__ part_s,
                           float* __restrict__ lse_t, int* __restrict__ counters,
                           int* __restrict__ rej, T* __restrict__ hrow,
                           int* __restrict__ out_tokens, int* __restrict__ n_acc,
                           int* __restrict__ n_emit, int* err) {
  __shared__ float red[kRowThreads / 32];
  __shared__ float redm[kRowThreads / 32];
  __shared__ int flag;
  __shared__ int nrej;
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x, row = blockIdx.y, nch = gridDim.x;
  const int b = row / S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* src = logits + (long long)row * V;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  // one pass: running (max, sum of exp((x - max) / tau)) per thread, 16-byte loads
  float mx = -INFINITY, s = 0.f;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(src + v0) & 15) == 0;
  const int nv = vec_ok ? (v1 - v0) / 8 : 0;
  for (int k = threadIdx.x; k < nv; k += kRowThreads) {
    float x[8];
    load8_stream(src + v0 + 8 * k, x);
    float lm = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                     fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
    if (lm > mx) {
      s = mx == -INFINITY ? 0.f : s * __expf((mx - lm) * inv_temp);
      mx = lm;
    }
    if (mx == -INFINITY) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += __expf((x[j] - mx) * inv_temp);
  }
  for (int v = v0 + 8 * nv + threadIdx.x; v < v1; v += kRowThreads) {
    const float x = to_f32<T>(src[v]);
    if (x > mx) {
      s = mx == -INFINITY ? 0.f : s * __expf((mx - x) * inv_temp);
      mx = x;
    }
    if (mx != -INFINITY) s += __expf((x - mx) * inv_temp);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_merge(mx, s, m2, s2, inv_temp);
  }
  if (lane == 0) {
    redm[warp] = mx;
    red[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mx = redm[0];
    s = red[0];
    for (int w = 1; w < kRowThreads / 32; ++w) ms_merge(mx, s, redm[w], red[w], inv_temp);
    part_m[(long long)row * nch + c] = mx;
    part_s[(long long)row * nch + c] = s;
  }
  // last chunk of this row -> the row's log-sum-exp
  if (!elect_last(&counters[row], nch, &flag)) return;
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int k = 0; k < nch; ++k) M = fmaxf(M, __ldcg(part_m + (long long)row * nch + k));
    float L = 0.f;
    for (int k = 0; k < nch; ++k)
      L += __ldcg(part_s + (long long)row * nch + k) *
           __expf((__ldcg(part_m + (long long)row * nch + k) - M) * inv_temp);
    lse_t[row] = M * inv_temp + logf(L);
  }
  // last row of the sequence -> acceptance walk
  const int seq_counter = gridDim.y + b;  // counters after the per-row ones
  if (!elect_last(&counters[seq_counter], S, &flag)) return;
  if (threadIdx.x == 0) {
    int n = 0;
    for (; n < S; ++n) {
      const long long r = (long long)b * S + n;
      const int dt = draft[r];
      if (dt < 0 || dt >= V) { raise_error(err, DFLASH_DEV_BAD_INDEX); break; }
      const float lp = to_f32<T>(logits[r * V + dt]) * inv_temp - __ldcg(lse_t + r);
      const float lq = dmax[r] * inv_temp - dlse[r];  // the draft is the drafter's argmax
      // accept iff u < p/q, compared as log u < log p - log q
      const float uu = u[r * 2];
      if (!(uu < __expf(lp - lq))) break;
      out_tokens[r] = dt;
    }
    for (int i = n; i < S; ++i) out_tokens[(long long)b * S + i] = -1;
    rej[b] = n;
    n_acc[b] = n;
    n_emit[b] = n < S ? n + 1 : S;
    nrej = n;
  }
  __syncthreads();
  const int rs = min(nrej, S - 1);
  for (int k = threadIdx.x; k < d; k += kRowThreads)
    hrow[(long long)b * d + k] = hidden[((long long)b * S + rs) * d + k];
}

// Pass 2, grid (chunks, B), after the drafter logits zr [B, V] of each rejected slot
// were recomputed: r_v = max(0, p_v - q_v) per chunk; the last chunk of a sequence
// finds the chunk holding u[n,1] * sum(r) and, inside it, the token: each thread sums
// a contiguous segment, one block scan of the segment sums places the target in one
// segment, and that thread walks it.  Rounding (the chunk sums and the walk add in
// different orders) can leave the target just past the last mass: then the last index
// with mass is taken.
template <typename T>
__device__ __forceinline__ float resid_val(const T* lt, const float* lz, int v, float it,
                                           float lset, float lsez, bool use_p) {
  const float p = __expf(to_f32<T>(lt[v]) * it - lset);
  const float q = __expf(lz[v] * it - lsez);
  return use_p ? p : fmaxf(0.f, p - q);
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads)
    k_verify_sample_residual(const T* __restrict__ logits, const float* __restrict__ zr,
                             const float* __restrict__ lse_t, const float* __restrict__ dlse,
                             const float* __restrict__ u, const int* __restrict__ rej, int S,
                             int V, int chunk, float inv_temp, float* __restrict__ part_r,
                             float* __restrict__ part_p, int* __restrict__ counters,
                             int* __restrict__ out_tokens) {
  __shared__ float red[kRowThreads / 32];
  __shared__ int flag;
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x, b = blockIdx.y, nch = gridDim.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = rej[b];
  if (n >= S) return;  // everything accepted: nothing to sample (counter unused)
  const long long r = (long long)b * S + n;
  const T* lt = logits + r * V;
  const float* lz = zr + (long long)b * V;
  const float lset = lse_t[r], lsez = dlse[r];
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  float sr = 0.f, sp = 0.f;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(lt + v0) | reinterpret_cast<uintptr_t>(lz + v0)) & 15) == 0;
  const int nv = vec_ok ? (v1 - v0) / 8 : 0;
  for (int k = threadIdx.x; k < nv; k += kRowThreads) {
    float x[8], z[8];
    load8(lt + v0 + 8 * k, x);
    load8(lz + v0 + 8 * k, z);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p = __expf(x[j] * inv_temp - lset);
      const float q = __expf(z[j] * inv_temp - lsez);
      sr += fmaxf(0.f, p - q);
      sp += p;
    }
  }
  for (int v = v0 + 8 * nv + threadIdx.x; v < v1; v += kRowThreads) {
    const float p = __expf(to_f32<T>(lt[v]) * inv_temp - lset);
    const float q = __expf(lz[v] * inv_temp - lsez);
    sr += fmaxf(0.f, p - q);
    sp += p;
  }
  sr = block_sum(sr, red);
  sp = block_sum(sp, red);
  if (threadIdx.x == 0) {
    part_r[(long long)b * nch + c] = sr;
    part_p[(long long)b * nch + c] = sp;
  }
  if (!elect_last(&counters[b], nch, &flag)) return;
  // choose the residual (or p itself when the residual is all zero), then the chunk
  __shared__ int use_p_s, cstar, found, lastnz;
  __shared__ float target_s, before_s;
  __shared__ float wtot[kRowThreads / 32];
  if (threadIdx.x == 0) {
    float Z = 0.f;
    for (int k = 0; k < nch; ++k) Z += __ldcg(part_r + (long long)b * nch + k);
    const float* pr = part_r;
    use_p_s = (Z <= 0.f);
    if (use_p_s) {
      Z = 0.f;
      for (int k = 0; k < nch; ++k) Z += __ldcg(part_p + (long long)b * nch + k);
      pr = part_p;
    }
    const float target = u[r * 2 + 1] * Z;
    float acc = 0.f;
    int k = 0, last_nz = -1;
    for (; k < nch; ++k) {
      const float w = __ldcg(pr + (long long)b * nch + k);
      if (w > 0.f) last_nz = k;
      if (acc + w >= target && w > 0.f) break;
      acc += w;
    }
    if (k == nch) {  // rounding: no prefix reached the target; the last mass is taken
      k = last_nz < 0 ? 0 : last_nz;
      acc = INFINITY;
    }
    cstar = k;
    before_s = acc;
    target_s = target;
    found = 0x7fffffff;
    lastnz = -1;
  }
  __syncthreads();
  const bool use_p = use_p_s != 0;
  const float target = target_s, before = before_s;
  const int w0 = cstar * chunk, w1 = min(V, w0 + chunk);
  const int seg = ((w1 - w0 + kRowThreads - 1) / kRowThreads + 7) & ~7;
  const int a0 = min(w1, w0 + threadIdx.x * seg), a1 = min(w1, a0 + seg);
  const bool seg_vec = ((reinterpret_cast<uintptr_t>(lt + a0) | reinterpret_cast<uintptr_t>(lz + a0)) & 15) == 0;
  float my = 0.f;
  int my_last = -1;
  int v = a0;
  if (seg_vec) {
    for (; v + 8 <= a1; v += 8) {
      float x[8], z[8];
      load8(lt + v, x);
      load8(lz + v, z);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p = __expf(x[j] * inv_temp - lset);
        const float q = __expf(z[j] * inv_temp - lsez);
        const float val = use_p ? p : fmaxf(0.f, p - q);
        my += val;
        if (val > 0.f) my_last = v + j;
      }
    }
  }
  for (; v < a1; ++v) {
    const float val = resid_val(lt, lz, v, inv_temp, lset, lsez, use_p);
    my += val;
    if (val > 0.f) my_last = v;
  }
  // exclusive scan of the segment sums in thread (= index) order
  float incl = my;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  float woff = 0.f;
  for (int w = 0; w < warp; ++w) woff += wtot[w];
  const float excl = woff + incl - my;
  const float lo = before + excl;
  const bool last_mass = !(before < INFINITY);
  if (!last_mass && my > 0.f && lo + my >= target && (lo < target || excl == 0.f)) {
    float acc = lo;
    int hit = my_last;   // the walk may fall just short through rounding
    for (int w = a0; w < a1; ++w) {
      const float val = resid_val(lt, lz, w, inv_temp, lset, lsez, use_p);
      acc += val;
      if (val > 0.f && acc >= target) {
        hit = w;
        break;
      }
    }
    atomicMin(&found, hit);
  }
  if (my_last >= 0) atomicMax(&lastnz, my_last);
  __syncthreads();
  if (threadIdx.x == 0) out_tokens[r] = found != 0x7fffffff ? found : lastnz;
}

// ------------------------------------------------------------- speculative loop
// Target input of the block: the anchor (slot 0 of block_ids) then drafts 1..S-1.
static __global__ void k_spec_target_ids(const int* __restrict__ block_ids,
                                         const int* __restrict__ draft, int M, int S,
                                         int* __restrict__ ids) {
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < M) ids[m] = (m % S == 0) ? block_ids[m] : draft[m];
}

// Synthetic agreement of the target with the drafter (a stand-in for a trained pair):
// row i < S-1 of sequence b gets logit[draft[b, i+1]] = max of the row + 1 when
// u[(step mod u_steps), b, i] < p.  grid (B*S), one CTA per row.
static __global__ void __launch_bounds__(kRowThreads)
    k_spec_plant(float* __restrict__ logits, const int* __restrict__ draft,
                 const float* __restrict__ u, int u_steps, const int* __restrict__ step,
                 float p, int S, int V, int M, int* err) {
  __shared__ float red[kRowThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int m = blockIdx.x, i = m % S;
  if (i == S - 1) return;
  const int st = (*step) % u_steps;
  if (!(u[(long long)st * M + m] < p)) return;
  const int d = draft[m + 1];
  if (d < 0 || d >= V) {
    if (threadIdx.x == 0) raise_error(err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  float* row = logits + (long long)m * V;
  float mx = -INFINITY;
  for (int v = threadIdx.x; v < V; v += kRowThreads) mx = fmaxf(mx, row[v]);
  mx = warp_max(mx);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = red[0];
    for (int w = 1; w < kRowThreads / 32; ++w) t = fmaxf(t, red[w]);
    row[d] = t + 1.0f;
  }
}

// Commit of one verified block per sequence (one thread per sequence): the drafter's
// injection positions and cache slots of the block's S rows (from the old context
// length), the emitted tokens appended to `generated`, the next block's ids (the last
// emitted token as the anchor, then mask ids) and the new context length; thread 0 of
// CTA 0 advances the step counter.
static __global__ void k_spec_commit(const int* __restrict__ out_tokens,
                                     const int* __restrict__ n_emit, int B, int S, int mask_id,
                                     int* __restrict__ block_ids, int* __restrict__ ctx_lens,
                                     const int* __restrict__ page_table, int max_pages,
                                     int* __restrict__ positions, int* __restrict__ slots,
                                     int* __restrict__ generated, int max_new,
                                     int* __restrict__ n_generated, int* __restrict__ step,
                                     int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0 && step) *step += 1;
  if (b >= B) return;
  const int ctx = ctx_lens[b];
  for (int i = 0; i < S; ++i) {
    const int p = ctx + i, pi = p / kPage;
    int page = 0;
    if (p < 0 || pi >= max_pages || (page = page_table[(long long)b * max_pages + pi]) < 0) {
      raise_error(err, DFLASH_DEV_BAD_INDEX);
      page = 0;
    }
    positions[b * S + i] = p;
    slots[b * S + i] = page * kPage + p % kPage;
  }
  const int ne = n_emit[b];
  if (ne < 1 || ne > S) {   // verification did not finish (its error is already set)
    raise_error(err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  const int g0 = n_generated[b];
  for (int i = 0; i < ne; ++i)
    if (g0 + i < max_new) generated[(long long)b * max_new + g0 + i] = out_tokens[b * S + i];
  n_generated[b] = min(max_new, g0 + ne);
  block_ids[b * S] = out_tokens[b * S + ne - 1];
  for (int i = 1; i < S; ++i) block_ids[b * S + i] = mask_id;
  ctx_lens[b] = ctx + ne;
}

}  // namespace dflash
