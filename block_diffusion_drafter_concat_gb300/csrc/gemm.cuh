// Weight-streaming GEMM  Y[M, N] = A[M, K] * W[N, K]^T  with fused epilogues.
//
// Every projection of the drafter step is one of these: the fused-feature projection,
// the injected K/V projections, Q/K/V, O, gate/up, down and the LM head.  At batch 1
// the block has 16 rows, so the contraction is a stream of weights past a small
// activation tile: the tensor-core kernel puts 128 weight rows on the MMA's M side and
// the activation rows on its N side (swap-AB), pulls 128x64 weight boxes and BNx64
// activation boxes into a shared-memory ring with TMA (128-byte swizzle, mbarrier
// completion), and runs ldmatrix + mma.sync.m16n8k16 (bf16 in, fp32 accumulate).
//
// Work is split "stream-K" style: the (m-block, n-tile, k-stage) units are cut into
// one contiguous range per persistent CTA, so every SM streams the same number of
// weight bytes whatever the shape.  A tile cut between CTAs is finished by the last
// contributor to count itself in, which sums the published partial tiles in contributor
// order (deterministic) and runs the epilogue; each contributor publishes its piece
// before it counts, so the finisher never waits.  Weight boxes of the first stages are issued
// before griddepcontrol.wait, overlapping the previous kernel's tail.
#pragma once

#include "common.cuh"

namespace dflash {

constexpr int kMaxSeg = 16;  // weight segments of one projection launch (K/V of up to 8 layers)

enum Epi : int {
  EPI_F32 = 0,    // y[m, n] = v (fp32)
  EPI_QKV = 1,    // segments q | k | v: RoPE on q and k, bf16 into attention layouts
  EPI_KV = 2,     // segments k0 | v0 | k1 | v1 ...: RoPE on k, scatter into cache pages
  EPI_RESID = 3,  // x[m, n] += v (fp32 residual stream)
  EPI_SWIGLU = 4, // paired tiles (64 gate rows | 64 up rows): act = silu(g) * u
  EPI_ARGMAX = 5, // per-tile (max, argmax, sum exp) of each row for the LM head
  EPI_ARGKEY = 6  // greedy LM head: per-row packed (max, argmax) keys, finished in-kernel
};

struct WMaps {
  CUtensorMap m[kMaxSeg];
};

template <typename T>
struct EpiArgs {
  int M, N;
  float* y;
  int ldy;
  // rotary / attention layouts
  const int* pos;
  const float2* rope;  // [max_position][head_dim/2] (cos, sin)
  int max_pos;
  int S, hq, hkv, hd;
  T* q;    // [B][hkv][S*G][hd]
  T* kb;   // [B][hkv][S][hd]
  T* vb;   // [B][hkv][S][hd]
  // cache injection
  T* kpool[kMaxSeg / 2];
  T* vpool[kMaxSeg / 2];
  const int* slots;
  long long num_slots;
  // SwiGLU
  T* act;
  int F;
  // LM-head argmax partials, [n_tiles][M]
  float* am_max;
  int* am_idx;
  float* am_sum;
  float inv_temp;
  int want_sum;
  // greedy LM head without partials: per-row packed keys (atomic maximum), a CTA
  // counter; the last CTA writes tokens (and max logits) and clears both
  unsigned long long* am_key;
  int* am_done;
  int* tok_out;
  float* max_out;
  // EPI_QKV: the last n_inj of the M rows are new context rows (fused target features):
  // their K (RoPE at inj_pos) and V go to the layer's cache pages at inj_slots, their Q
  // is not stored
  int n_inj;
  const int* inj_pos;
  const int* inj_slots;
  T* inj_kpool;
  T* inj_vpool;
  int* err;
};

struct GemmShape {
  int M, K, n_tiles, ks, m_blocks, paired, nseg;
  int bn;          // activation rows per tile
  int tile_mode;   // 1: CTAs take whole tiles (no split); 0: stream-K unit ranges
  int pair;        // tcgen05 whole tiles on SM pairs (two weight tiles per pair)
  long long units;
  int seg_tile0[kMaxSeg + 1];
  int seg_rows[kMaxSeg];  // rows of each weight matrix
  float* part;      // [grid][2][BN * kBM] partial tiles (split pieces)
  int* counters;    // one per output tile
  // wait_extra is 0 except under the forced-timeout test hook, which makes the finisher
  // of a split tile wait, for at most wait_ns, for one count more than can arrive (the
  // tcgen05 kernel's finisher waits for contributors - 1 + wait_extra publications)
  int wait_extra;
  unsigned long long wait_ns;
  // FP8 weights (k_gemm_tc<..., true>): per-segment row scales, applied to each
  // contribution as it leaves the accumulators (null for bf16 / fp32 weights)
  const float* wscale[kMaxSeg];
};

// ---------------------------------------------------------------------------- epilogue
// Cs: the finished fp32 tile, Cs[r * pitch + c] for activation row m0 + r and output
// column c of n-tile nt.  Runs on `nthr` threads (thread index `tid`, whole warps).
// Each warp takes whole rows (r = warp, warp + nw, ...) and its lanes the columns, so
// the integer work of a row (sequence, slot, position) is done once per row, every
// global access of a warp is contiguous, and the loads of four rows are issued before
// the first of their stores.
template <typename T>
__device__ __forceinline__ void store_pair(T* p, float a, float b) {
  if constexpr (sizeof(T) == 2) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(a, b);
  } else {
    *reinterpret_cast<float2*>(p) = make_float2(a, b);
  }
}

template <typename T, int EPI>
__device__ void tile_epilogue(const float* Cs, int pitch, int BN, int m0, int nt,
                              const GemmShape& g, const EpiArgs<T>& e, int tid, int nthr) {
  int seg = 0;
  while (seg + 1 < g.nseg && nt >= g.seg_tile0[seg + 1]) ++seg;
  const int rows_per_tile = g.paired ? kBM / 2 : kBM;
  const int r0 = (nt - g.seg_tile0[seg]) * rows_per_tile;  // first row within the segment
  const int mr = min(BN, e.M - m0);
  const int lane = tid & 31, warp = tid >> 5, nw = nthr >> 5;
  constexpr int RB = 4;  // rows per batch of a warp

  if constexpr (EPI == EPI_F32 || EPI == EPI_RESID) {
    const int nc = min(kBM, e.N - nt * kBM);
    if ((nc & 3) == 0 && (e.ldy & 3) == 0 && (pitch & 3) == 0) {
      // lane -> columns 4*lane .. 4*lane+3 (lanes past a ragged last tile's columns idle)
      const int rlim = 4 * lane < nc ? mr : 0;
      for (int rb = warp; rb < rlim; rb += nw * RB) {
        float4 o[RB];
        if constexpr (EPI == EPI_RESID) {
#pragma unroll
          for (int k = 0; k < RB; ++k) {
            const int r = rb + k * nw;
            if (r < mr)
              o[k] = reinterpret_cast<const float4*>(e.y + (long long)(m0 + r) * e.ldy + nt * kBM)[lane];
          }
        }
#pragma unroll
        for (int k = 0; k < RB; ++k) {
          const int r = rb + k * nw;
          if (r >= mr) continue;
          float4 v = *reinterpret_cast<const float4*>(Cs + r * pitch + lane * 4);
          if constexpr (EPI == EPI_RESID) {
            v.x += o[k].x; v.y += o[k].y; v.z += o[k].z; v.w += o[k].w;
          }
          reinterpret_cast<float4*>(e.y + (long long)(m0 + r) * e.ldy + nt * kBM)[lane] = v;
        }
      }
    } else {
      for (int r = warp; r < mr; r += nw) {
        float* yr = e.y + (long long)(m0 + r) * e.ldy + nt * kBM;
        for (int c = lane; c < nc; c += 32) {
          const float v = Cs[r * pitch + c];
          if constexpr (EPI == EPI_RESID) yr[c] += v; else yr[c] = v;
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // 64 gate columns and the 64 matching up columns; lane -> columns 2*lane, 2*lane+1
    const int f = r0 + 2 * lane;
    const bool pair_ok = ((e.F & 1) == 0) && f + 1 < e.F;
    for (int r = warp; r < mr; r += nw) {
      T* ar = e.act + (long long)(m0 + r) * e.F;
      const float2 gt = *reinterpret_cast<const float2*>(Cs + r * pitch + 2 * lane);
      const float2 up = *reinterpret_cast<const float2*>(Cs + r * pitch + 64 + 2 * lane);
      const float a0 = gt.x / (1.0f + __expf(-gt.x)) * up.x;
      const float a1 = gt.y / (1.0f + __expf(-gt.y)) * up.y;
      if (pair_ok) {
        store_pair<T>(ar + f, a0, a1);
      } else {
        if (f < e.F) ar[f] = from_f32<T>(a0);
        if (f + 1 < e.F) ar[f + 1] = from_f32<T>(a1);
      }
    }
  } else if constexpr (EPI == EPI_QKV || EPI == EPI_KV) {
    const int hd = e.hd, half = hd >> 1;
    // segment kind: 0 = q, 1 = k, 2 = v
    int kind, layer = 0;
    if constexpr (EPI == EPI_QKV) kind = seg;
    else { layer = seg >> 1; kind = 1 + (seg & 1); }
    const int G = e.hq / e.hkv;
    const int nheads = (kind == 0) ? e.hq : e.hkv;
    if (kind == 2) {
      // lane -> columns 2*lane + 64*k (k = 0, 1): head and offset fixed per lane
      int hv[2], jv[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int f = r0 + 2 * lane + 64 * k;
        hv[k] = f / hd;
        jv[k] = f - hv[k] * hd;
      }
      for (int rb = warp; rb < mr; rb += nw * RB) {
        long long rbase[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int r = rb + q * nw;
          rbase[q] = -1;
          if (r >= mr) continue;
          const int m = m0 + r;
          int slot = -1;
          bool pool = EPI == EPI_KV;
          if constexpr (EPI == EPI_QKV) {
            if (m >= e.M - e.n_inj) {
              pool = true;
              slot = e.inj_slots[m - (e.M - e.n_inj)];
            }
          } else {
            slot = e.slots[m];
          }
          if (pool) {
            if (slot < 0 || slot >= e.num_slots) { raise_error(e.err, DFLASH_DEV_BAD_INDEX); continue; }
            rbase[q] = ((long long)(slot / kPage) * e.hkv * kPage + slot % kPage) * hd;  // + head*16*hd
            if constexpr (EPI == EPI_QKV) rbase[q] |= 1LL << 62;   // marks a cache row
          } else {
            const int b = m / e.S, ii = m - (m / e.S) * e.S;
            rbase[q] = ((long long)b * e.hkv * e.S + ii) * hd;   // + head * S * hd
          }
        }
#pragma unroll
        for (int q = 0; q < RB; ++q) {
          const int r = rb + q * nw;
          if (r >= mr || rbase[q] < 0) continue;
          const bool to_pool = EPI == EPI_KV || (rbase[q] >> 62) != 0;
          const long long base = rbase[q] & ((1LL << 62) - 1);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (hv[k] >= e.hkv) continue;
            const float2 v = *reinterpret_cast<const float2*>(Cs + r * pitch + 2 * lane + 64 * k);
            if (to_pool) {
              T* vp;
              if constexpr (EPI == EPI_QKV) vp = e.inj_vpool; else vp = e.vpool[layer];
              store_pair<T>(vp + base + (long long)hv[k] * kPage * hd + jv[k], v.x, v.y);
            } else {
              store_pair<T>(e.vb + base + (long long)hv[k] * e.S * hd + jv[k], v.x, v.y);
            }
          }
        }
      }
    } else {
      // rotary pairs (j, j + hd/2) of one head lie in the same 128-column tile; lane ->
      // the adjacent pair indices 2*lane and 2*lane + 1 of the tile's 64 pairs when half
      // head_dim is even (one head: results stored as pairs), else lane and lane + 32
      const bool adj = (half & 1) == 0;
      int cv[2], hv[2], jv[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int cc = adj ? 2 * lane + k : lane + 32 * k;
        const int hl = cc / half;
        jv[k] = cc - hl * half;
        cv[k] = hl * hd + jv[k];
        hv[k] = (r0 + cv[k]) / hd;
      }
      // rows in batches of 8 per warp: lane q < 8 fetches row q's position (and cache
      // slot), shuffles broadcast them, then the 16 rotary-table loads of the batch go
      // out together: two dependent round trips per 8 rows
      constexpr int RR = 8;
      for (int rb = warp; rb < mr; rb += nw * RR) {
        int my_p = -1;
        long long my_base = 0;
        int my_inj = 0;
        if (lane < RR) {
          const int r = rb + lane * nw;
          if (r < mr) {
            const int m = m0 + r;
            const bool inj = EPI == EPI_QKV && m >= e.M - e.n_inj;   // a new context row
            const int p = inj ? e.inj_pos[m - (e.M - e.n_inj)] : e.pos[m];
            bool ok = p >= 0 && p < e.max_pos;
            if (!ok) raise_error(e.err, DFLASH_DEV_BAD_POSITION);
            if (inj) {
              const int slot = e.inj_slots[m - (e.M - e.n_inj)];
              if (kind == 0) {
                ok = false;                                   // its Q is not needed
              } else if (slot < 0 || slot >= e.num_slots) {
                raise_error(e.err, DFLASH_DEV_BAD_INDEX);
                ok = false;
              } else {
                my_base = ((long long)(slot / kPage) * e.hkv * kPage + slot % kPage) * hd;
                my_inj = 1;
              }
            } else if constexpr (EPI == EPI_QKV) {
              const int b = m / e.S, ii = m - (m / e.S) * e.S;
              my_base = kind == 0 ? (((long long)b * e.hkv * e.S + ii) * G) * hd   // + (gk*S*G + hh)*hd
                                  : ((long long)b * e.hkv * e.S + ii) * hd;        // + head*S*hd
            } else {
              const int slot = e.slots[m];
              if (slot < 0 || slot >= e.num_slots) {
                raise_error(e.err, DFLASH_DEV_BAD_INDEX);
                ok = false;
              } else {
                my_base = ((long long)(slot / kPage) * e.hkv * kPage + slot % kPage) * hd;
              }
            }
            if (ok) my_p = p;
          }
        }
        int pv[RR], injv[RR];
        long long rbase[RR];
#pragma unroll
        for (int q = 0; q < RR; ++q) {
          pv[q] = __shfl_sync(0xffffffffu, my_p, q);
          rbase[q] = __shfl_sync(0xffffffffu, my_base, q);
          injv[q] = __shfl_sync(0xffffffffu, my_inj, q);
        }
        float2 cs[RR][2];
#pragma unroll
        for (int q = 0; q < RR; ++q) {
          if (adj) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (pv[q] >= 0) v = *reinterpret_cast<const float4*>(e.rope + (long long)pv[q] * half + jv[0]);
            cs[q][0] = make_float2(v.x, v.y);
            cs[q][1] = make_float2(v.z, v.w);
          } else {
#pragma unroll
            for (int k = 0; k < 2; ++k)
              cs[q][k] = pv[q] >= 0 ? e.rope[(long long)pv[q] * half + jv[k]] : make_float2(0.f, 0.f);
          }
        }
        auto dst_of = [&](int head, long long base, int to_cache) -> T* {
          if constexpr (EPI == EPI_QKV) {
            if (to_cache) return e.inj_kpool + base + (long long)head * kPage * hd;
            if (kind == 0) {
              const int gk = head / G, hh = head - gk * G;
              return e.q + base + ((long long)gk * e.S * G + hh) * hd;
            }
            return e.kb + base + (long long)head * e.S * hd;
          } else {
            return e.kpool[layer] + base + (long long)head * kPage * hd;
          }
        };
#pragma unroll
        for (int q = 0; q < RR; ++q) {
          const int r = rb + q * nw;
          if (pv[q] < 0) continue;   // past the chunk, or reported above
          float y0[2], y1[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float x0 = Cs[r * pitch + cv[k]], x1 = Cs[r * pitch + cv[k] + half];
            y0[k] = x0 * cs[q][k].x - x1 * cs[q][k].y;
            y1[k] = x1 * cs[q][k].x + x0 * cs[q][k].y;
          }
          if (adj) {
            if (hv[0] >= nheads) continue;   // both indices belong to head hv[0]
            T* dst = dst_of(hv[0], rbase[q], injv[q]);
            store_pair<T>(dst + jv[0], y0[0], y0[1]);
            store_pair<T>(dst + jv[0] + half, y1[0], y1[1]);
          } else {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              if (hv[k] >= nheads) continue;
              T* dst = dst_of(hv[k], rbase[q], injv[q]);
              dst[jv[k]] = from_f32<T>(y0[k]);
              dst[jv[k] + half] = from_f32<T>(y1[k]);
            }
          }
        }
      }
    }
  } else if constexpr (EPI == EPI_ARGMAX || EPI == EPI_ARGKEY) {
    // Four threads per row, every row of the chunk at once (a warp per row would walk
    // its rows one after another, each behind a five-level shuffle chain).  Thread
    // `sub` of a row takes columns sub, sub + 4, ... (conflict-free: the four threads
    // and eight rows of a warp hit 32 distinct banks), then (max, lowest index) and the
    // sum of exponentials are merged over the row's four threads with two shuffles.
    const int nc = min(kBM, e.N - nt * kBM);
    const int sub = tid & 3;
    for (int rb = 0; rb < mr; rb += nthr >> 2) {
      const int r = rb + (tid >> 2);
      const bool active = r < mr;
      float best = -INFINITY;
      int bi = 0x7fffffff;
      if (active) {
#pragma unroll 8
        for (int j = 0; j < kBM / 4; ++j) {
          const int c = sub + 4 * j;
          if (c < nc) {
            const float v = Cs[r * pitch + c];
            if (v > best) { best = v; bi = nt * kBM + c; }
          }
        }
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
      }
      if constexpr (EPI == EPI_ARGMAX) {
        float sum = 0.f;
        if (e.want_sum) {
          if (active) {
#pragma unroll 8
            for (int j = 0; j < kBM / 4; ++j) {
              const int c = sub + 4 * j;
              if (c < nc) sum += __expf((Cs[r * pitch + c] - best) * e.inv_temp);
            }
          }
          sum += __shfl_xor_sync(0xffffffffu, sum, 1);
          sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        }
        if (active && sub == 0) {
          const long long o = (long long)nt * e.M + m0 + r;
          e.am_max[o] = best;
          e.am_idx[o] = bi;
          e.am_sum[o] = sum;
        }
      } else {
        if (active && sub == 0) atomicMax(e.am_key + m0 + r, argmax_key(best, bi));
      }
    }
  }
}

// ------------------------------------------------------------- tensor-core kernel
// A pipeline stage: a 128-row weight box and the matching activation box(es).  bf16
// weights: 64 k per stage (128 x 128 B); FP8 weights: 128 k per stage (128 x 128 B of
// e4m3 codes) and two 64-k activation boxes.
template <int BN, bool F8 = false>
struct TcCfg {
  static constexpr int KS = F8 ? 2 * kBK : kBK;          // k per stage
  // FP8: two CTAs per SM (two consumer warps per scheduler hide the conversions'
  // latency), so each holds a shorter ring (3 and 2 stages: 606 -> 598 us a batch-1
  // step against 4 and 3; 2/2: 615, 3/3: 600).  bf16: rings of 8 (16 rows) and 6 (32
  // rows) stages leave room on the SM for a CTA of the next kernels (attention, RMSNorm,
  // combine) to start while the projection drains: measured on GB300 at batch 1,
  // 718 -> 708 us a step against 10 and 8 stages (9/6: 713, 8/7: 712, 6/5: 709, 5/4: 734).
  static constexpr int NS = F8 ? (BN == 16 ? 3 : 2)
                               : (BN == 16 ? 8 : BN == 32 ? 6 : BN == 64 ? 6 : 4);
  static constexpr int CTAS_PER_SM = F8 ? 2 : 1;
  static constexpr int W_BYTES = kBM * kBK * 2;           // 16 KB either way
  static constexpr int A_BYTES = BN * KS * 2;
  static constexpr int STAGE = W_BYTES + A_BYTES;
  static constexpr int PITCH = kBM + 4;
  static constexpr int CS_BYTES = BN * PITCH * 4;
  static constexpr int MAXC = 512;  // contributors of one tile (units per CTA >= 4)
  static constexpr int SMEM = 1024 /*align slack*/ + NS * STAGE + CS_BYTES + 2 * NS * 8 + 16 +
                              MAXC * 4;
  static constexpr int THREADS = 160;  // 4 consumer warps + 1 TMA producer warp
};

// Publication of a CTA's partial tile: after a CTA barrier one thread's release-add
// makes every thread's earlier writes visible at GPU scope to an acquiring reader.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Counting in after publishing: release orders this CTA's earlier writes (after a CTA
// barrier) before the add, acquire makes the other counted CTAs' writes visible.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Range of units [u0, u1) of CTA c out of `grid`.
__device__ __forceinline__ void cta_range(long long units, int c, int grid, long long& u0,
                                          long long& u1) {
  u0 = units * c / grid;
  u1 = units * (c + 1) / grid;
}

// Contributors of tile t (units [t*ks, (t+1)*ks)): the CTAs whose non-empty unit range
// intersects it, in CTA order.  Writes each one's partial slot (cta*2 + 0 when its range
// starts inside the tile, + 1 when the tile is the last piece of its range) to `slots`
// when given, and returns how many there are.  With at least one unit per CTA the
// contributors are the consecutive CTAs [c_lo, c_hi] found with two divisions (this
// runs on the tail of every split tile, so it must stay cheap).
__device__ __forceinline__ int tile_contributors(long long units, int grid, int ks, int t,
                                                 int* slots) {
  const long long ts = static_cast<long long>(t) * ks, te = ts + ks;
  // CTA c owns [units*c/grid, units*(c+1)/grid): c_lo is the last CTA starting at or
  // before ts, c_hi the last starting before te
  const int c_lo = static_cast<int>(((ts + 1) * grid + units - 1) / units) - 1;
  const int c_hi = static_cast<int>((te * grid + units - 1) / units) - 1;
  if (units >= grid) {
    if (slots) {
      slots[0] = c_lo * 2 + ((units * c_lo / grid == ts) ? 0 : 1);
      for (int c = c_lo + 1; c <= c_hi; ++c) slots[c - c_lo] = c * 2;
    }
    return c_hi - c_lo + 1;
  }
  int n = 0;  // fewer units than CTAs: skip the CTAs with empty ranges
  for (int c = c_lo; c <= c_hi; ++c) {
    const long long s0 = units * c / grid, s1 = units * (c + 1) / grid;
    if (s1 <= ts || s0 == s1) continue;
    if (slots) slots[n] = c * 2 + ((s0 / ks == t) ? 0 : 1);
    ++n;
  }
  return n;
}

// Incremental walk over (m-block, n-tile, k-stage) units for the TMA producer:
// coordinates of the weight box (segment, row, k) and the activation box (m-block).
struct UnitWalk {
  int ks, nt, mb, seg, row;
  __device__ __forceinline__ void locate(const GemmShape& g) {
    seg = 0;
    while (seg + 1 < g.nseg && nt >= g.seg_tile0[seg + 1]) ++seg;
    row = g.paired ? nt * (kBM / 2) : (nt - g.seg_tile0[seg]) * kBM;
  }
  __device__ __forceinline__ void start(const GemmShape& g, long long u) {
    const int t = static_cast<int>(u / g.ks);
    ks = static_cast<int>(u - static_cast<long long>(t) * g.ks);
    mb = t / g.n_tiles;
    nt = t - mb * g.n_tiles;
    locate(g);
  }
  __device__ __forceinline__ void next(const GemmShape& g) {
    if (++ks < g.ks) return;
    ks = 0;
    if (++nt == g.n_tiles) { nt = 0; ++mb; }
    locate(g);
  }
};

// Scale of weight row `wr` (0..127) of n-tile nt: its segment's row scale (paired
// tiles: 64 rows of segment 0 then the same 64 rows of segment 1).  Rows past a
// segment's end (zero-filled boxes) take 0.
__device__ __forceinline__ float tile_row_scale(const GemmShape& g, int nt, int wr) {
  int seg = 0, row;
  if (g.paired) {
    seg = wr >> 6;
    row = nt * (kBM / 2) + (wr & 63);
  } else {
    while (seg + 1 < g.nseg && nt >= g.seg_tile0[seg + 1]) ++seg;
    row = (nt - g.seg_tile0[seg]) * kBM + wr;
  }
  return row < g.seg_rows[seg] ? __ldg(g.wscale[seg] + row) : 0.f;
}

__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// Two e4m3 codes of a 32-bit word (bytes lo and lo + 1, the lower first) as an f16 pair
// holding value * 2^-8, by integer bit placement: the code's exponent and mantissa bits
// (eeee mmm) become the f16's low exponent and high mantissa bits and its sign the f16
// sign.  e4m3 (bias 7) and f16 (bias 15) both read exponent field 0 as 0.mmm at the
// lowest normal exponent, so normal and subnormal codes alike come out as exactly
// value * 2^-8 (the scale carries the 2^8).  No conversion-pipe instruction is used.
// Three instructions per pair: a byte permute puts each code in the low byte of a 16-bit
// half with its sign replicated into the high byte, a shift by 7 moves the exponent and
// mantissa bits into place (and a replicated sign bit to bit 15 of the half), and a mask
// keeps exactly those bits.
template <int LO>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t word) {
  uint32_t t;   // halves: byte LO | sign(byte LO) x 8, byte LO + 1 | sign(byte LO + 1) x 8
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(word), "n"(LO == 0 ? 0x9180 : 0xB3A2));
  return (t << 7) & 0xBF80BF80u;
}
// A bf16 pair as an f16 pair (round to nearest; exact in f16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Greedy LM head: after this CTA's epilogues, count it; the last CTA of the grid turns
// the rows' packed keys into tokens (and max logits) and clears keys and counter.
template <typename T, typename Sync>
__device__ __forceinline__ void argmax_keys_finish(const EpiArgs<T>& e, int M, int tid, int nthr,
                                                   int* flag, Sync sync) {
  sync();
  if (tid == 0) {
    __threadfence();
    flag[0] = (atomicAdd(e.am_done, 1) == static_cast<int>(gridDim.x) - 1);
  }
  sync();
  if (!flag[0]) return;
  __threadfence();
  for (int m = tid; m < M; m += nthr) {
    float v;
    int idx;
    argmax_unkey(atomicExch(e.am_key + m, 0ull), v, idx);
    e.tok_out[m] = idx;
    if (e.max_out) e.max_out[m] = v;
  }
  if (tid == 0) *e.am_done = 0;
}

// F8 = true: the weights are FP8 e4m3 codes with per-row scales (g.wscale); the MMA
// runs on f16 operands: the codes as value * 2^-8 (exact, e4m3x2_to_f16x2_scaled) and
// the bf16 activations converted to f16 (exact but for values below 2^-14, whose few
// lowest bits f16 subnormals drop); the accumulators are scaled by 2^8 * s_n.  Within every 32-k chunk the
// k index is permuted alike for both operands so that a lane reads 8 consecutive weight
// bytes and 8 consecutive activations: MMA 1 takes k 8t..8t+3, MMA 2 k 8t+4..8t+7 of
// lane group t (the contraction sums over every k once either way).
template <int BN, int EPI, bool F8 = false>
__global__ void __launch_bounds__(160, F8 ? 2 : 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ WMaps wm,
              const GemmShape g, const EpiArgs<bf16> e) {
  using C = TcCfg<BN, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* Cs = reinterpret_cast<float*>(smem + C::NS * C::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::NS * C::STAGE + C::CS_BYTES);
  uint64_t* empty = full + C::NS;
  int* flag = reinterpret_cast<int*>(empty + C::NS);
  int* cslot = flag + 4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  long long u0, u1;
  cta_range(g.units, cta, grid, u0, u1);
  const int n_my = static_cast<int>(u1 - u0);

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // The single issuing thread must keep up with HBM (one 16 KB weight box every
      // ~0.3 us per SM), so the unit walk is incremental: no division per unit.
      tma_prefetch_desc(&tmA);
      const uint64_t pol = policy_evict_first();
      UnitWalk wc, ac;
      wc.start(g, u0);
      ac = wc;
      // weight boxes are 128 bytes wide: 64 bf16 or 128 e4m3 values of k
      auto issue_w = [&](int s, const UnitWalk& w) {
        uint8_t* st = stages + s * C::STAGE;
        if (g.paired) {
          tma_load_2d_hint(st, &wm.m[0], &full[s], w.ks * C::KS, w.row, pol);
          tma_load_2d_hint(st + C::W_BYTES / 2, &wm.m[1], &full[s], w.ks * C::KS, w.row, pol);
        } else {
          tma_load_2d_hint(st, &wm.m[w.seg], &full[s], w.ks * C::KS, w.row, pol);
        }
      };
      // activation boxes are 128 bytes wide: 64 bf16 values of k, two per FP8 stage
      auto issue_a = [&](int s, const UnitWalk& w) {
        uint8_t* at = stages + s * C::STAGE + C::W_BYTES;
#pragma unroll
        for (int j = 0; j < C::KS / kBK; ++j)
          tma_load_2d(at + j * BN * 128, &tmA, &full[s], w.ks * C::KS + j * kBK, w.mb * BN);
      };
      const int pre = min(C::NS, n_my);
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], C::STAGE);
        issue_w(i, wc);
        wc.next(g);
      }
      pdl_wait();  // activations are written by the previous kernel
      for (int i = 0; i < pre; ++i) {
        issue_a(i, ac);
        ac.next(g);
      }
      int issued = pre;
      int s = pre % C::NS;
      uint32_t par = (pre / C::NS) & 1;  // parity of this stage's current use
      for (int i = pre; i < n_my; ++i) {
        if (!mbar_wait(&empty[s], par ^ 1)) {
          raise_error(e.err, DFLASH_DEV_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE);
        issue_w(s, wc);
        issue_a(s, ac);
        wc.next(g);
        ac.next(g);
        issued = i + 1;
        if (++s == C::NS) { s = 0; par ^= 1; }
      }
      // never leave with copies in flight
      for (int i = max(0, issued - C::NS); i < issued; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  constexpr int NB = BN / 8;  // n8 tiles of activation rows
  float acc[2][NB][4];
  const int g8 = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
  bool ok = true;
  long long u = u0;
  int i = 0;
  while (u < u1) {
    const int t = static_cast<int>(u / g.ks);
    const int ks0 = static_cast<int>(u % g.ks);
    const long long tile_end = static_cast<long long>(t + 1) * g.ks;
    const long long seg_end = min(tile_end, u1);
    const int nk = static_cast<int>(seg_end - u);
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;
    for (int k = 0; k < nk; ++k, ++i) {
      const int s = i % C::NS;
      // After a timeout the warp keeps walking the same units and barriers (without
      // waiting or computing) so that no named barrier is left short of a warp.
      if (ok && !__all_sync(0xffffffffu, mbar_wait(&full[s], (i / C::NS) & 1))) {
        if (lane == 0) raise_error(e.err, DFLASH_DEV_TIMEOUT);
        ok = false;
      }
      if (!ok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      const uint32_t wbase = smem_u32(stages + s * C::STAGE);
      const uint32_t abase = wbase + C::W_BYTES;
      if constexpr (F8) {
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
          uint32_t a1[2][4], a2[2][4];
#pragma unroll
          for (int ms = 0; ms < 2; ++ms) {
            const int row = warp * 32 + ms * 16 + g8;
            const uint32_t off = ((kc * 32 + 8 * t4) & 15);
            const uint2 w0 = lds_u2(wbase + swz128(row, kc * 2 + (t4 >> 1)) + off);
            const uint2 w1 = lds_u2(wbase + swz128(row + 8, kc * 2 + (t4 >> 1)) + off);
            a1[ms][0] = e4m3x2_to_f16x2_scaled<0>(w0.x);
            a1[ms][1] = e4m3x2_to_f16x2_scaled<0>(w1.x);
            a1[ms][2] = e4m3x2_to_f16x2_scaled<2>(w0.x);
            a1[ms][3] = e4m3x2_to_f16x2_scaled<2>(w1.x);
            a2[ms][0] = e4m3x2_to_f16x2_scaled<0>(w0.y);
            a2[ms][1] = e4m3x2_to_f16x2_scaled<0>(w1.y);
            a2[ms][2] = e4m3x2_to_f16x2_scaled<2>(w0.y);
            a2[ms][3] = e4m3x2_to_f16x2_scaled<2>(w1.y);
          }
          // activations: box kc / 2, 16-byte chunk (kc % 2) * 4 + t of row nb * 8 + g8
          const uint32_t ab = abase + (kc >> 1) * (BN * 128);
#pragma unroll
          for (int nb = 0; nb < BN / 8; ++nb) {
            const uint4 v = lds_u4(ab + swz128(nb * 8 + g8, (kc & 1) * 4 + t4));
            const uint32_t h0 = bf16x2_to_f16x2(v.x), h1 = bf16x2_to_f16x2(v.y);
            const uint32_t h2 = bf16x2_to_f16x2(v.z), h3 = bf16x2_to_f16x2(v.w);
#pragma unroll
            for (int ms = 0; ms < 2; ++ms) {
              mma_f16(acc[ms][nb], a1[ms], h0, h1);
              mma_f16(acc[ms][nb], a2[ms], h2, h3);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[2][4];
#pragma unroll
        for (int ms = 0; ms < 2; ++ms) {
          int row = warp * 32 + ms * 16 + (mi & 1) * 8 + r8;
          ldsm_x4(a[ms], wbase + swz128(row, kk * 2 + (mi >> 1)));
        }
#pragma unroll
        for (int nb = 0; nb < BN / 16; ++nb) {
          uint32_t b[4];
          int row = nb * 16 + (mi >> 1) * 8 + r8;
          ldsm_x4(b, abase + swz128(row, kk * 2 + (mi & 1)));
#pragma unroll
          for (int ms = 0; ms < 2; ++ms) {
            mma_bf16(acc[ms][nb * 2 + 0], a[ms], b[0], b[1]);
            mma_bf16(acc[ms][nb * 2 + 1], a[ms], b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // ---- tile (or piece of tile) done (FP8: accumulators times the row scales)
    if constexpr (F8) {
      const int ntl = t % g.n_tiles;
#pragma unroll
      for (int ms = 0; ms < 2; ++ms) {
        const float s0 = 256.f * tile_row_scale(g, ntl, warp * 32 + ms * 16 + g8);
        const float s1 = 256.f * tile_row_scale(g, ntl, warp * 32 + ms * 16 + g8 + 8);
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          acc[ms][j][0] *= s0; acc[ms][j][1] *= s0;
          acc[ms][j][2] *= s1; acc[ms][j][3] *= s1;
        }
      }
    }
    const bool whole = (ks0 == 0) && (seg_end == tile_end);
    bool mine = true;
    if (!whole) {
      // A tile split between CTAs.  Every contributor publishes its piece (in the
      // accumulators' own fragment layout: each (ms, j) fragment of the 128 threads is
      // 2 KB contiguous) and then counts itself in with one acquire-release add; the
      // last to count finishes the tile, summing the pieces in contributor order, its
      // own from registers.  Every piece is published before its count, so the
      // finisher never waits.
      int* arrived = g.counters + t;
      const int slot = (u == u0) ? 0 : 1;
      float4* dst = reinterpret_cast<float4*>(g.part + ((long long)cta * 2 + slot) * BN * kBM);
#pragma unroll
      for (int ms = 0; ms < 2; ++ms)
#pragma unroll
        for (int j = 0; j < NB; ++j)
          dst[(ms * NB + j) * 128 + tid] =
              make_float4(acc[ms][j][0], acc[ms][j][1], acc[ms][j][2], acc[ms][j][3]);
      consumer_sync();
      if (tid == 0) {
        const int nc = tile_contributors(g.units, grid, g.ks, t, cslot);
        const bool last = atom_add_acq_rel_gpu(arrived, 1) == nc - 1;
        if (last && g.wait_extra) {
          // forced-timeout test hook: wait, boundedly, for one arrival more than can come
          const unsigned long long t0 = global_ns();
          while (ld_acquire_gpu(arrived) < nc + g.wait_extra) {
            if (global_ns() - t0 > g.wait_ns) {
              raise_error(e.err, DFLASH_DEV_TIMEOUT);
              break;
            }
          }
        }
        if (last) *arrived = 0;   // every contributor has counted: free for the next launch
        flag[0] = last;
        flag[1] = nc;
      }
      consumer_sync();
      mine = flag[0] != 0;
      if (mine) {
        // the loads of CR contributors' pieces are in flight together
        const int nc = flag[1];
        constexpr int XN = 2 * NB;
        constexpr int CR = XN >= 16 ? 1 : 16 / XN;
        float4 sum[XN];
#pragma unroll
        for (int q = 0; q < XN; ++q) sum[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c0 = 0; c0 < nc; c0 += CR) {
          float4 v[CR][XN];
#pragma unroll
          for (int jc = 0; jc < CR; ++jc) {
            if (c0 + jc >= nc) continue;
            const int cs = cslot[c0 + jc];
            const float4* src = reinterpret_cast<const float4*>(g.part + (long long)cs * BN * kBM);
#pragma unroll
            for (int q = 0; q < XN; ++q) {
              if ((cs >> 1) == cta) {
                v[jc][q] = make_float4(acc[q / NB][q % NB][0], acc[q / NB][q % NB][1],
                                       acc[q / NB][q % NB][2], acc[q / NB][q % NB][3]);
              } else {
                v[jc][q] = __ldcg(src + q * 128 + tid);
              }
            }
          }
#pragma unroll
          for (int jc = 0; jc < CR; ++jc) {
            if (c0 + jc >= nc) continue;
#pragma unroll
            for (int q = 0; q < XN; ++q) {
              sum[q].x += v[jc][q].x; sum[q].y += v[jc][q].y;
              sum[q].z += v[jc][q].z; sum[q].w += v[jc][q].w;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < XN; ++q) {
          acc[q / NB][q % NB][0] = sum[q].x; acc[q / NB][q % NB][1] = sum[q].y;
          acc[q / NB][q % NB][2] = sum[q].z; acc[q / NB][q % NB][3] = sum[q].w;
        }
      }
    }
    if (mine) {
      // accumulators -> Cs[activation row][output column]
#pragma unroll
      for (int ms = 0; ms < 2; ++ms)
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const int wr = warp * 32 + ms * 16 + g8;
          const int ar = j * 8 + 2 * t4;
          Cs[ar * C::PITCH + wr] = acc[ms][j][0];
          Cs[(ar + 1) * C::PITCH + wr] = acc[ms][j][1];
          Cs[ar * C::PITCH + wr + 8] = acc[ms][j][2];
          Cs[(ar + 1) * C::PITCH + wr + 8] = acc[ms][j][3];
        }
      consumer_sync();
    }
    if (mine) {
      const int mb = t / g.n_tiles, nt = t % g.n_tiles;
      tile_epilogue<bf16, EPI>(Cs, C::PITCH, BN, mb * BN, nt, g, e, tid, 128);
    }
    consumer_sync();
    u = seg_end;
  }
  if constexpr (EPI == EPI_ARGKEY) argmax_keys_finish(e, g.M, tid, 128, flag, consumer_sync);
}

// ------------------------------------------------------------------- fp32 SIMT kernel
// fp32 workloads keep full fp32 products (no TF32): one CTA per (m-block, n-tile) of
// 16 rows x 128 columns, FFMA over K, then the same epilogues.
constexpr int kF32BN = 16;
constexpr int kF32BK = 64;

struct WPtrs {
  const float* p[kMaxSeg];
};

template <int EPI>
__global__ void __launch_bounds__(256)
    k_gemm_f32(const float* __restrict__ A, int lda, const WPtrs Wseg, const GemmShape g,
               const EpiArgs<float> e) {
  __shared__ float As[kF32BN][kF32BK + 1];
  __shared__ float Ws[kBM][kF32BK + 1];
  __shared__ __align__(16) float Cs[kF32BN * (kBM + 4)];
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int mb = t / g.n_tiles, nt = t % g.n_tiles;
  int seg = 0;
  while (seg + 1 < g.nseg && nt >= g.seg_tile0[seg + 1]) ++seg;
  const int tid = threadIdx.x;
  const int rows_per_tile = g.paired ? kBM / 2 : kBM;
  const int r0 = (nt - g.seg_tile0[seg]) * rows_per_tile;
  // thread -> (act row ar, 8 weight rows wr..wr+7 strided by 16)
  const int ar = tid % kF32BN, wr0 = tid / kF32BN;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // The next k-tile is loaded into registers while this one is multiplied from shared
  // memory (the loop is a chain of global round trips otherwise); k stays in ascending
  // order, so the sums are those of the plain loop.
  constexpr int NA = kF32BN * kF32BK / 256, NW = kBM * kF32BK / 256;
  float ra[NA], rw[NW];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int q = 0; q < NA; ++q) {
      const int x = tid + q * 256, r = x / kF32BK, k = x % kF32BK;
      const int m = mb * kF32BN + r;
      ra[q] = (m < g.M && k0 + k < g.K) ? A[(long long)m * lda + k0 + k] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int x = tid + q * 256, r = x / kF32BK, k = x % kF32BK;
      const int sg = g.paired ? (r < kBM / 2 ? 0 : 1) : seg;
      const int row = r0 + (g.paired ? r % (kBM / 2) : r);
      rw[q] = (row < g.seg_rows[sg] && k0 + k < g.K) ? Wseg.p[sg][(long long)row * g.K + k0 + k]
                                                       : 0.f;
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < g.K; k0 += kF32BK) {
#pragma unroll
    for (int q = 0; q < NA; ++q) {
      const int x = tid + q * 256;
      As[x / kF32BK][x % kF32BK] = ra[q];
    }
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int x = tid + q * 256;
      Ws[x / kF32BK][x % kF32BK] = rw[q];
    }
    __syncthreads();
    if (k0 + kF32BK < g.K) fetch(k0 + kF32BK);
#pragma unroll 4
    for (int k = 0; k < kF32BK; ++k) {
      float a = As[ar][k];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(a, Ws[wr0 + 16 * j][k], acc[j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) Cs[ar * (kBM + 4) + wr0 + 16 * j] = acc[j];
  __syncthreads();
  tile_epilogue<float, EPI>(Cs, kBM + 4, kF32BN, mb * kF32BN, nt, g, e, tid, 256);
}

}  // namespace dflash
