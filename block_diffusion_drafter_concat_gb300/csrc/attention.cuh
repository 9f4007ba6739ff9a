// Block attention of the drafter over the paged context cache plus the block itself.
//
// For sequence b and kv head g the S*G query rows (block slot i, q head g*G + hh, row
// i*G + hh) attend, with no mask, to the sequence's ctx_len cached context keys
// (injected target features) followed by the block's own S keys (with `causal`, slot i
// sees the block keys 0..i only: chunks of new context run through the layer stack).  Keys are walked a
// 16-token page at a time; the work of one (b, g) is split over CTAs by contiguous
// ranges of pages (split-context, "flash-decoding"), each CTA keeps an online softmax
// (running max in the log2 domain, running sum, unnormalised output) and publishes
// it; a combine kernel merges the splits in split order and writes the attention output
// in [B*S, hq*hd] layout for the output projection (a single split writes it directly).
//
// bf16 kernel: K and V pages arrive by TMA (two-dimensional view of the pool,
// 16 x 64 boxes, 128-byte swizzle) in a ring of mbarrier-tracked stages; QK^T and PV
// run on mma.sync.m16n8k16 with the probabilities re-used from the score registers
// (as a bf16 hi/lo pair).
#pragma once

#include "common.cuh"

namespace dflash {

template <typename T>
struct AttnArgs {
  const T* q;        // [B][hkv][QR][hd]
  const T* kb;       // [B][hkv][S][hd]  (fp32 path reads these directly)
  const T* vb;
  const T* kpool;    // fp32 path: the layer's pools
  const T* vpool;
  const int* page_table;
  int max_pages;
  const int* ctx_lens;
  int num_pages;
  int S, hq, hkv, hd, QR;
  int pps;           // key pages per split
  int nsplit;
  float* part_o;     // [B][hkv][nsplit][QR][hd]
  float* part_ml;    // [B][hkv][nsplit][QR][2]
  T* out;            // [B*S][hq*hd]
  int* err;
  // 0: every query row sees all S block keys (the drafter's block); 1: query row r
  // (block slot r / G) sees block keys 0..r / G only (a causal chunk of new context or
  // target tokens)
  int causal;
  // the newest `fresh` context positions of every sequence were written by the
  // predecessor kernel (context rows injected by the Q/K/V projection): their pages are
  // fetched after the wait, not before (0: every context page predates it)
  int fresh;
};

// Tensor maps of the tcgen05 attention kernel: q as [B*hkv*QR, hd] with 128-row boxes,
// the pools and the block K/V with 16-row boxes.
struct AuMaps {
  CUtensorMap q, k, v, kb, vb;
  CUtensorMap po;   // split partial O as fp32 rows [.., hd], boxes of QR rows x 32 columns
};

struct AttnMaps {
  CUtensorMap k, v, kb, vb;
};

// Combine of the published splits, grid (ceil(QR / 8), hkv, B), 8 rows x hd/4 threads:
// out[r] = sum_s w_s o_s / sum_s w_s l_s with w_s = 2^(m_s - max m), splits in order.
// SF: splits whose loads are in flight at once (16 for many splits; 4 or 8 when a launch
// has at most that many, where the registers of 16 would only cut the occupancy).  The splits are
// merged one after another in either case, so SF does not change the result.
template <typename T, int SF>
__global__ void __launch_bounds__(256) k_attn_combine(const AttnArgs<T> a) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.z, g = blockIdx.y;
  const int hd4 = a.hd / 4;
  const int r = blockIdx.x * 8 + threadIdx.x / hd4, d4 = threadIdx.x % hd4;
  if (r >= a.QR) return;
  const int ctx = a.ctx_lens[b];
  if (ctx < 0 || ctx > a.max_pages * kPage) return;   // reported by the attention kernel
  const int kp = (ctx + kPage - 1) / kPage + 1;
  const int ns = (kp + a.pps - 1) / a.pps;
  const long long grp = (long long)b * a.hkv + g;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + grp * a.nsplit * a.QR;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + grp * a.nsplit * a.QR * a.hd);
  // one pass in split order with a running maximum (loads of SF splits in flight)
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += SF) {
    float4 v[SF];
    float2 q[SF];
#pragma unroll
    for (int j = 0; j < SF; ++j)
      if (s0 + j < ns) {
        q[j] = ml[(long long)(s0 + j) * a.QR + r];
        v[j] = po[((long long)(s0 + j) * a.QR + r) * hd4 + d4];
      }
#pragma unroll
    for (int j = 0; j < SF; ++j)
      if (s0 + j < ns) {
        const float nm = fmaxf(M, q[j].x);
        const float al = exp2f(M - nm), w = exp2f(q[j].x - nm);
        M = nm;
        L = L * al + w * q[j].y;
        acc.x = acc.x * al + w * v[j].x;
        acc.y = acc.y * al + w * v[j].y;
        acc.z = acc.z * al + w * v[j].z;
        acc.w = acc.w * al + w * v[j].w;
      }
  }
  const float inv = 1.f / L;
  const int G = a.hq / a.hkv, i = r / G, hh = r % G;
  T* dst = a.out + ((long long)b * a.S + i) * (a.hq * a.hd) + (g * G + hh) * a.hd + d4 * 4;
  dst[0] = from_f32<T>(acc.x * inv);
  dst[1] = from_f32<T>(acc.y * inv);
  dst[2] = from_f32<T>(acc.z * inv);
  dst[3] = from_f32<T>(acc.w * inv);
}

// A split's online-softmax state: with one split the output is final and written
// directly, otherwise (o unnormalised, m, l) go to the partial buffers.
template <typename T>
__device__ __forceinline__ void attn_emit(const AttnArgs<T>& a, int b, int g, int split, int r,
                                          int d, float o0, float o1, float l) {
  const long long grp = (long long)b * a.hkv + g;
  if (a.nsplit == 1) {
    const float inv = 1.f / l;
    const int G = a.hq / a.hkv, i = r / G, hh = r % G;
    T* out = a.out + ((long long)b * a.S + i) * (a.hq * a.hd) + (g * G + hh) * a.hd + d;
    out[0] = from_f32<T>(o0 * inv);
    out[1] = from_f32<T>(o1 * inv);
  } else {
    float* po = a.part_o + ((grp * a.nsplit + split) * a.QR + r) * a.hd + d;
    *reinterpret_cast<float2*>(po) = make_float2(o0, o1);
  }
}

// ------------------------------------------------------------------ bf16 tensor core
constexpr int kAttnStages = 8;

// Shared memory of the mma.sync attention kernel: the K/V ring and its barriers.
__host__ __device__ constexpr int attn_tc_smem(int hd) {
  return 1024 + kAttnStages * (2 * kPage * hd * 2 + 16) + 16;
}

template <int HD>
struct AttnCfg {
  static constexpr int NS = kAttnStages;
  static constexpr int TILE = kPage * HD * 2;   // one K (or V) page of one head
  static constexpr int STAGE = 2 * TILE;
  static constexpr int MAXSPLIT = 64;
};

template <int HD, int NW>
__global__ void __launch_bounds__((NW + 1) * 32)
    k_attn_tc(const __grid_constant__ AttnMaps maps, const AttnArgs<bf16> a) {
  using C = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NS * C::STAGE);
  uint64_t* empty = full + C::NS;

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Context lengths, the page table and the context pages were written before the
  // previous kernel started: they are read, and the context pages fetched, before the
  // wait.  Only q and the block's own K/V come from the previous kernel.
  const int T = a.ctx_lens[b];
  if (T < 0 || T > a.max_pages * kPage) {
    if (tid == 0) raise_error(a.err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  const int np = (T + kPage - 1) / kPage;   // context pages
  const int kp = np + 1;                    // + the block's own keys
  const int ns = (kp + a.pps - 1) / a.pps;
  if (split >= ns) return;                  // this split is past the sequence's keys
  const int p0 = split * a.pps, p1 = min(kp, p0 + a.pps);
  const int nmy = p1 - p0;
  // stages fetched before the wait: context pages that predate the predecessor, within
  // the first ring
  const int fresh_pg = a.fresh > 0 ? max(0, T - a.fresh) / kPage : np;
  const int pre = max(0, min(C::NS, min(np, fresh_pg) - p0));

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == NW) {
    // The page ids of this split are read 32 at a time by the whole warp (one round
    // trip) and handed to lane 0, which issues the TMA copies.
    int issued = 0;
    bool ok = true;
    for (int base = 0; base < nmy && ok; base += 32) {
      int my_page = 0;
      const int pgl = p0 + base + lane;
      if (base + lane < nmy && pgl < np) my_page = a.page_table[(long long)b * a.max_pages + pgl];
      const int cnt = min(32, nmy - base);
      for (int j = 0; j < cnt; ++j) {
        const int page_j = __shfl_sync(0xffffffffu, my_page, j);
        const int i = base + j;
        // the block's own keys, fresh pages, and stages beyond the first ring follow
        // the wait
        if (i == pre) pdl_wait();
        if (lane == 0 && ok) {
          const int s = i % C::NS;
          if (i >= C::NS && !mbar_wait(&empty[s], ((i / C::NS) - 1) & 1)) {
            raise_error(a.err, DFLASH_DEV_TIMEOUT);
            ok = false;
          } else {
            mbar_arrive_expect_tx(&full[s], C::STAGE);
            uint8_t* kd = stages + s * C::STAGE;
            uint8_t* vd = kd + C::TILE;
            const int pg = p0 + i;
            const CUtensorMap *mk, *mv;
            int row;
            if (pg < np) {
              int page = page_j;
              if (page < 0 || page >= a.num_pages) {
                raise_error(a.err, DFLASH_DEV_BAD_INDEX);
                page = 0;
              }
              mk = &maps.k; mv = &maps.v;
              row = (page * a.hkv + g) * kPage;
            } else {
              mk = &maps.kb; mv = &maps.vb;
              row = (b * a.hkv + g) * a.S;
            }
#pragma unroll
            for (int bx = 0; bx < HD / 64; ++bx) {
              tma_load_2d(kd + bx * 2048, mk, &full[s], bx * 64, row);
              tma_load_2d(vd + bx * 2048, mv, &full[s], bx * 64, row);
            }
            issued = i + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (lane == 0)
      for (int i = max(0, issued - C::NS); i < issued; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1);
  } else {
    // ------------------------------------------------------------------ consumers
    pdl_wait();   // q is written by the previous kernel
    pdl_launch_dependents();
    const int g8 = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
    const int qr0 = warp * 16;
    const bf16* qb = a.q + (((long long)b * a.hkv + g) * a.QR + qr0) * HD;
    uint32_t qf[HD / 16][4];
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      qf[kk][0] = *reinterpret_cast<const uint32_t*>(qb + (g8)*HD + kk * 16 + 2 * t4);
      qf[kk][1] = *reinterpret_cast<const uint32_t*>(qb + (g8 + 8) * HD + kk * 16 + 2 * t4);
      qf[kk][2] = *reinterpret_cast<const uint32_t*>(qb + (g8)*HD + kk * 16 + 8 + 2 * t4);
      qf[kk][3] = *reinterpret_cast<const uint32_t*>(qb + (g8 + 8) * HD + kk * 16 + 8 + 2 * t4);
    }
    float o[HD / 8][4];
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sc = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    for (int i = 0; i < nmy; ++i) {
      const int s = i % C::NS;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / C::NS) & 1))) {
        if (lane == 0) raise_error(a.err, DFLASH_DEV_TIMEOUT);
        break;
      }
      const int pg = p0 + i;
      const int valid = (pg < np) ? min(kPage, T - pg * kPage) : a.S;
      const bool cmask = a.causal && pg >= np;   // block keys past the row's own slot
      const uint32_t kbase = smem_u32(stages + s * C::STAGE);
      const uint32_t vbase = kbase + C::TILE;
      float sacc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t kf[4];
        const int key = (mi >> 1) * 8 + r8;
        const int ch = kk * 2 + (mi & 1);
        ldsm_x4(kf, kbase + (ch >> 3) * 2048 + swz128(key, ch & 7));
        mma_bf16(sacc[0], qf[kk], kf[0], kf[1]);
        mma_bf16(sacc[1], qf[kk], kf[2], kf[3]);
      }
      // mask keys past `valid` (only a page's last keys can be), row max on raw scores
      // (the scale is positive), then scale and reference in one FMA per key: the log2
      // domain probabilities 2^(s*sc - m)
      if (valid < kPage || cmask) {
        const int G = a.hq / a.hkv;
        const int slot0 = cmask ? (qr0 + g8) / G : kPage, slot1 = cmask ? (qr0 + g8 + 8) / G : kPage;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int key = n * 8 + 2 * t4 + (c & 1);
            if (key >= valid || key > (c < 2 ? slot0 : slot1)) sacc[n][c] = -INFINITY;
          }
      }
      float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
      float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float nm0 = fmaxf(m0, mx0 * sc), nm1 = fmaxf(m1, mx1 * sc);
      const float al0 = exp2f(m0 - nm0), al1 = exp2f(m1 - nm1);
      m0 = nm0;
      m1 = nm1;
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        p[n][0] = exp2f(fmaf(sacc[n][0], sc, -nm0));
        p[n][1] = exp2f(fmaf(sacc[n][1], sc, -nm0));
        p[n][2] = exp2f(fmaf(sacc[n][2], sc, -nm1));
        p[n][3] = exp2f(fmaf(sacc[n][3], sc, -nm1));
      }
      l0 = l0 * al0 + p[0][0] + p[0][1] + p[1][0] + p[1][1];
      l1 = l1 * al1 + p[0][2] + p[0][3] + p[1][2] + p[1][3];
#pragma unroll
      for (int j = 0; j < HD / 8; ++j) {
        o[j][0] *= al0; o[j][1] *= al0;
        o[j][2] *= al1; o[j][3] *= al1;
      }
      // P as a bf16 pair hi + lo: a single bf16 P would put a 2^-9 relative error on
      // the output (a sum of zero-mean terms, so it does not average out); the pair
      // keeps it near 2^-17 for a second MMA per tile.
      uint32_t pa[4], pl[4];
      split_bf16x2(p[0][0], p[0][1], pa[0], pl[0]);
      split_bf16x2(p[0][2], p[0][3], pa[1], pl[1]);
      split_bf16x2(p[1][0], p[1][1], pa[2], pl[2]);
      split_bf16x2(p[1][2], p[1][3], pa[3], pl[3]);
#pragma unroll
      for (int dj = 0; dj < HD / 16; ++dj) {
        uint32_t vf[4];
        const int key = (mi & 1) * 8 + r8;
        const int ch = dj * 2 + (mi >> 1);
        ldsm_x4_trans(vf, vbase + (ch >> 3) * 2048 + swz128(key, ch & 7));
        mma_bf16(o[2 * dj], pa, vf[0], vf[1]);
        mma_bf16(o[2 * dj + 1], pa, vf[2], vf[3]);
        mma_bf16(o[2 * dj], pl, vf[0], vf[1]);
        mma_bf16(o[2 * dj + 1], pl, vf[2], vf[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      const int d = j * 8 + 2 * t4;
      attn_emit<bf16>(a, b, g, split, qr0 + g8, d, o[j][0], o[j][1], l0);
      attn_emit<bf16>(a, b, g, split, qr0 + g8 + 8, d, o[j][2], o[j][3], l1);
    }
    if (t4 == 0 && a.nsplit > 1) {
      const long long grp = (long long)b * a.hkv + g;
      float* pm = a.part_ml + ((grp * a.nsplit + split) * a.QR + qr0) * 2;
      pm[g8 * 2] = m0;
      pm[g8 * 2 + 1] = l0;
      pm[(g8 + 8) * 2] = m1;
      pm[(g8 + 8) * 2 + 1] = l1;
    }
  }
}

// ---------------------------------------------------------------------- fp32 path
// Plain FFMA attention for fp32 workloads (small shapes), same splits and combine.
static __global__ void __launch_bounds__(128) k_attn_f32(const AttnArgs<float> a) {
  extern __shared__ float sm[];
  const int QR = a.QR, hd = a.hd;
  float* Qs = sm;                    // [QR][hd]
  float* Os = Qs + QR * hd;          // [QR][hd]
  float* Ks = Os + QR * hd;          // [16][hd]
  float* Vs = Ks + kPage * hd;       // [16][hd]
  float* Ss = Vs + kPage * hd;       // [QR][16]
  float* mrow = Ss + QR * kPage;     // [QR]
  float* lrow = mrow + QR;
  float* arow = lrow + QR;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  const int T = a.ctx_lens[b];
  if (T < 0 || T > a.max_pages * kPage) {
    if (tid == 0) raise_error(a.err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  const int np = (T + kPage - 1) / kPage, kp = np + 1;
  const int ns = (kp + a.pps - 1) / a.pps;
  if (split >= ns) return;
  const int p0 = split * a.pps, p1 = min(kp, p0 + a.pps);
  const long long grp = (long long)b * a.hkv + g;
  for (int x = tid; x < QR * hd; x += 128) {
    Qs[x] = a.q[grp * QR * hd + x];
    Os[x] = 0.f;
  }
  for (int r = tid; r < QR; r += 128) { mrow[r] = -INFINITY; lrow[r] = 0.f; }
  const float sc = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
  __syncthreads();
  for (int pg = p0; pg < p1; ++pg) {
    int valid;
    const float *ksrc, *vsrc;
    if (pg < np) {
      int page = a.page_table[(long long)b * a.max_pages + pg];
      if (page < 0 || page >= a.num_pages) {
        if (tid == 0) raise_error(a.err, DFLASH_DEV_BAD_INDEX);
        page = 0;
      }
      valid = min(kPage, T - pg * kPage);
      ksrc = a.kpool + ((long long)page * a.hkv + g) * kPage * hd;
      vsrc = a.vpool + ((long long)page * a.hkv + g) * kPage * hd;
    } else {
      valid = a.S;
      ksrc = a.kb + grp * a.S * hd;
      vsrc = a.vb + grp * a.S * hd;
    }
    for (int x = tid; x < kPage * hd; x += 128) {
      bool in = x / hd < valid;
      Ks[x] = in ? ksrc[x] : 0.f;
      Vs[x] = in ? vsrc[x] : 0.f;
    }
    __syncthreads();
    for (int x = tid; x < QR * kPage; x += 128) {
      int r = x / kPage, k = x % kPage;
      float s = 0.f;
      for (int d = 0; d < hd; ++d) s = fmaf(Qs[r * hd + d], Ks[k * hd + d], s);
      const bool seen = k < valid && !(a.causal && pg >= np && k > r / (a.hq / a.hkv));
      Ss[x] = seen ? s * sc : -INFINITY;
    }
    __syncthreads();
    for (int r = tid; r < QR; r += 128) {
      float mx = mrow[r];
      for (int k = 0; k < kPage; ++k) mx = fmaxf(mx, Ss[r * kPage + k]);
      float al = exp2f(mrow[r] - mx), sum = 0.f;
      for (int k = 0; k < kPage; ++k) {
        float p = exp2f(Ss[r * kPage + k] - mx);
        Ss[r * kPage + k] = p;
        sum += p;
      }
      lrow[r] = lrow[r] * al + sum;
      mrow[r] = mx;
      arow[r] = al;
    }
    __syncthreads();
    for (int x = tid; x < QR * hd; x += 128) {
      int r = x / hd, d = x % hd;
      float acc = Os[x] * arow[r];
      for (int k = 0; k < kPage; ++k) acc = fmaf(Ss[r * kPage + k], Vs[k * hd + d], acc);
      Os[x] = acc;
    }
    __syncthreads();
  }
  for (int x = tid; x < QR * hd; x += 128) {
    const int r = x / hd;
    if (a.nsplit == 1) {
      const int G = a.hq / a.hkv, i = r / G, hh = r % G, d = x % hd;
      a.out[((long long)b * a.S + i) * (a.hq * hd) + (g * G + hh) * hd + d] = Os[x] / lrow[r];
    } else {
      a.part_o[(grp * a.nsplit + split) * QR * hd + x] = Os[x];
    }
  }
  if (a.nsplit > 1) {
    float* pm = a.part_ml + (grp * a.nsplit + split) * QR * 2;
    for (int r = tid; r < QR; r += 128) { pm[2 * r] = mrow[r]; pm[2 * r + 1] = lrow[r]; }
  }
}

}  // namespace dflash
