// The drafter's layer stack as one persistent kernel for small blocks (batch x block
// <= 16 rows), one CTA per SM.
//
// At batch 1 each projection streams 8-300 MB of weights in a few microseconds, so
// separate kernels would spend much of the step in ramp-up, split-K tails and launch
// gaps.  Here every CTA walks the same list of phases -- per layer: Q/K/V (+RoPE),
// attention, split combine, output projection (+residual), RMSNorm, gate/up (+SwiGLU),
// down (+residual), RMSNorm -- separated by grid-wide barriers (bounded spins on a
// counter; the launch is cooperative so all CTAs are resident).  The TMA producer warp
// runs ahead across phases: weight boxes of the next projection (and context K/V pages
// of the next attention) are issued while the consumers are still in the previous
// phase or waiting at the barrier; only the activation boxes wait for the barrier.
// The projections reuse the stream-K schedule, MMA loop and epilogues of gemm.cuh and
// the attention math of attention.cuh.
#pragma once

#include "attention.cuh"
#include "gemm.cuh"

namespace dflash {

constexpr int kPMaxLayers = 8;
constexpr int kPMaxPhases = 8 * kPMaxLayers;
constexpr int kPNS = 10;                         // ring stages
constexpr int kPStage = kBM * kBK * 2 + 16 * kBK * 2;  // 16 KB weights + 2 KB activations
constexpr int kPHD = 128;                        // head_dim of this kernel
constexpr int kPQR = 64;                         // query rows per (sequence, kv head)
constexpr int kPPitch = kBM + 4;
constexpr int kPMaxC = 512;
constexpr int kPSmem = 1024 + kPNS * kPStage + 16 * kPPitch * 4 + 2 * kPNS * 8 + 64 + kPMaxC * 4;

enum PhaseType : int { PH_GEMM = 0, PH_ATTN = 1, PH_COMBINE = 2, PH_NORM = 3 };

struct PPhase {
  int type, epi, layer;
  int K, n_tiles, ks, nseg, paired;
  long long units;
  int seg_tile0[4];
  int seg_rows[4];
  int wmap[3];    // indices into PersistMaps::m (the paired tile uses wmap[0], wmap[1])
  int amap;       // activation map index
  int final_norm; // PH_NORM: final RMSNorm into final_hidden
};

// maps: per layer q, k, v, o, gate, up, down, kpool, vpool (index 9*l + j), then the
// activations n, o, act and the block k, v.
struct PersistMaps {
  CUtensorMap m[9 * kPMaxLayers + 5];
};
constexpr int kMapN = 9 * kPMaxLayers, kMapO = kMapN + 1, kMapAct = kMapN + 2,
              kMapKb = kMapN + 3, kMapVb = kMapN + 4;

struct PersistArgs {
  int n_phases, n_layers, d, qw, kvw, F, hq, hkv, S, B, M;
  PPhase ph[kPMaxPhases];
  // attention
  const int* ctx_lens;
  const int* page_table;
  int max_pages, num_pages, pps, nsplit;
  float* part_o;
  float* part_ml;
  // activations
  float* x;
  bf16* n;
  bf16* q;
  bf16* kb;
  bf16* vb;
  bf16* o;
  bf16* act;
  bf16* final_hidden;
  const int* pos;
  const float2* rope;
  int max_pos;
  const bf16* g_attn[kPMaxLayers];
  const bf16* g_mlp[kPMaxLayers];
  const bf16* g_final;
  float eps;
  float* part;     // stream-K partial tiles [grid][2][16][128]
  int* counters;   // tile counters
  int* bar;        // [0] barrier arrivals, [1] exits
  int* err;
};

#ifdef DFLASH_PERSIST_KERNEL  // the kernel is compiled in tu_persist.cu only
// ------------------------------------------------------------------ grid barrier
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until `*ctr >= target`; gives up after kWaitNs (raises DFLASH_DEV_TIMEOUT and
// returns so the kernel winds down instead of hanging).
__device__ __forceinline__ void grid_wait(const int* ctr, int target, int* err) {
  if (ld_acquire(ctr) >= target) return;
  const unsigned long long t0 = global_ns();
  while (ld_acquire(ctr) < target) {
    __nanosleep(64);
    if (global_ns() - t0 > kWaitNs) {
      raise_error(err, DFLASH_DEV_TIMEOUT);
      return;
    }
  }
}

// ------------------------------------------------------------------ unit iterator
// Walks the ring units of one CTA in order: stream-K units of the projections and the
// key pages of the attention items it owns (item i of a phase belongs to CTA i % grid).
struct PIter {
  int p;            // phase
  long long u, u1;  // projection units
  int item, pg, p1, np, b, g;  // attention: item, page, end page, context pages
  bool done;
};

__device__ __forceinline__ bool attn_item(const PersistArgs& a, int item, int& b, int& g,
                                          int& p0, int& p1, int& np) {
  const int per_b = a.hkv * a.nsplit;
  b = item / per_b;
  const int r = item % per_b;
  g = r / a.nsplit;
  const int split = r % a.nsplit;
  int T = a.ctx_lens[b];
  if (T < 0 || T > a.max_pages * kPage) T = 0;  // reported by the consumers
  np = (T + kPage - 1) / kPage;
  const int kp = np + 1;
  p0 = split * a.pps;
  p1 = min(kp, p0 + a.pps);
  return p0 < p1;
}

// Positions the iterator on the first ring unit at or after phase p.
__device__ void piter_enter(const PersistArgs& a, PIter& it, int p, int cta, int grid) {
  for (; p < a.n_phases; ++p) {
    const PPhase& ph = a.ph[p];
    if (ph.type == PH_GEMM) {
      it.u = ph.units * cta / grid;
      it.u1 = ph.units * (cta + 1) / grid;
      if (it.u < it.u1) { it.p = p; it.done = false; return; }
    } else if (ph.type == PH_ATTN) {
      const int items = a.B * a.hkv * a.nsplit;
      for (int item = cta; item < items; item += grid) {
        int b, g, p0, p1, np;
        if (attn_item(a, item, b, g, p0, p1, np)) {
          it.item = item; it.pg = p0; it.p1 = p1; it.np = np; it.b = b; it.g = g;
          it.p = p;
          it.done = false;
          return;
        }
      }
    }
  }
  it.done = true;
  it.p = a.n_phases;
}

__device__ void piter_next(const PersistArgs& a, PIter& it, int cta, int grid) {
  const PPhase& ph = a.ph[it.p];
  if (ph.type == PH_GEMM) {
    if (++it.u < it.u1) return;
  } else {
    if (++it.pg < it.p1) return;
    const int items = a.B * a.hkv * a.nsplit;
    for (int item = it.item + grid; item < items; item += grid) {
      int b, g, p0, p1, np;
      if (attn_item(a, item, b, g, p0, p1, np)) {
        it.item = item; it.pg = p0; it.p1 = p1; it.np = np; it.b = b; it.g = g;
        return;
      }
    }
  }
  piter_enter(a, it, it.p + 1, cta, grid);
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(160, 1)
    k_draft_persist(const __grid_constant__ PersistMaps maps, const __grid_constant__ PersistArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  float* Cs = reinterpret_cast<float*>(smem + kPNS * kPStage);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPNS * kPStage + 16 * kPPitch * 4);
  uint64_t* empty = full + kPNS;
  int* flag = reinterpret_cast<int*>(empty + kPNS);
  float* red = reinterpret_cast<float*>(flag + 4);  // 8 floats
  int* cslot = flag + 16;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < kPNS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 4) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      PIter wi, ai;
      bool waited = false;
      // the attention phases read the caller's context lengths: only after the wait
      if (a.ph[0].type != PH_GEMM || a.ph[0].units < grid) { pdl_wait(); waited = true; }
      piter_enter(a, wi, 0, cta, grid);
      ai = wi;
      long long wcount = 0, acount = 0;
      int bar_seen = 0;
      unsigned long long idle_since = 0;
      while (!ai.done) {
        bool did = false;
        // dependent part (activation box / block K,V) of the oldest issued unit
        if (acount < wcount) {
          const int need = ai.p * grid;
          bool ready;
          if (ai.p == 0) {
            if (!waited) { pdl_wait(); waited = true; }
            ready = true;
          } else {
            ready = bar_seen >= need;  // refreshed below only when nothing else can move
          }
          if (ready) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const int s = static_cast<int>(acount % kPNS);
            uint8_t* st = stages + s * kPStage;
            const PPhase& ph = a.ph[ai.p];
            if (ph.type == PH_GEMM) {
              const int ks = static_cast<int>(ai.u % ph.ks);
              tma_load_2d(st + kBM * kBK * 2, &maps.m[ph.amap], &full[s], ks * kBK, 0);
            } else if (ai.pg == ai.np) {  // the block's own keys
              const int row = (ai.b * a.hkv + ai.g) * a.S;
              tma_load_2d(st, &maps.m[kMapKb], &full[s], 0, row);
              tma_load_2d(st + 2048, &maps.m[kMapKb], &full[s], 64, row);
              tma_load_2d(st + 4096, &maps.m[kMapVb], &full[s], 0, row);
              tma_load_2d(st + 6144, &maps.m[kMapVb], &full[s], 64, row);
            }
            piter_next(a, ai, cta, grid);
            ++acount;
            did = true;
          }
        }
        // independent part (weight box / context K,V page) of the next unit
        if (!did && !wi.done) {
          const int s = static_cast<int>(wcount % kPNS);
          const long long k = wcount / kPNS;
          const PPhase& ph = a.ph[wi.p];
          const bool needs_inputs = ph.type == PH_ATTN;  // context pages need the cache
          if ((k == 0 || mbar_test_wait(&empty[s], static_cast<uint32_t>((k - 1) & 1))) &&
              (!needs_inputs || waited)) {
            uint8_t* st = stages + s * kPStage;
            if (ph.type == PH_GEMM) {
              mbar_arrive_expect_tx(&full[s], kPStage);
              const int t = static_cast<int>(wi.u / ph.ks), ks = static_cast<int>(wi.u % ph.ks);
              const int nt = t % ph.n_tiles;
              if (ph.paired) {
                const int row = nt * (kBM / 2);
                tma_load_2d_hint(st, &maps.m[ph.wmap[0]], &full[s], ks * kBK, row, pol);
                tma_load_2d_hint(st + kBM * kBK, &maps.m[ph.wmap[1]], &full[s], ks * kBK, row, pol);
              } else {
                int seg = 0;
                while (seg + 1 < ph.nseg && nt >= ph.seg_tile0[seg + 1]) ++seg;
                const int row = (nt - ph.seg_tile0[seg]) * kBM;
                tma_load_2d_hint(st, &maps.m[ph.wmap[seg]], &full[s], ks * kBK, row, pol);
              }
            } else {
              mbar_arrive_expect_tx(&full[s], 2 * kPage * kPHD * 2);
              if (wi.pg < wi.np) {
                int page = a.page_table[(long long)wi.b * a.max_pages + wi.pg];
                if (page < 0 || page >= a.num_pages) {
                  raise_error(a.err, DFLASH_DEV_BAD_INDEX);
                  page = 0;
                }
                const int row = (page * a.hkv + wi.g) * kPage;
                const CUtensorMap* mk = &maps.m[9 * ph.layer + 7];
                const CUtensorMap* mv = &maps.m[9 * ph.layer + 8];
                tma_load_2d(st, mk, &full[s], 0, row);
                tma_load_2d(st + 2048, mk, &full[s], 64, row);
                tma_load_2d(st + 4096, mv, &full[s], 0, row);
                tma_load_2d(st + 6144, mv, &full[s], 64, row);
              }
            }
            if (!waited && wi.p == 0 && wi.u + 1 == wi.u1) { pdl_wait(); waited = true; }
            piter_next(a, wi, cta, grid);
            ++wcount;
            did = true;
          }
        }
        if (!did && acount < wcount && ai.p > 0) {
          // weights are issued as far as the ring allows; now look at the barrier
          const int need = ai.p * grid;
          if ((bar_seen = ld_acquire(&a.bar[0])) >= need) continue;
        }
        if (did) {
          idle_since = 0;
        } else {
          const unsigned long long now = global_ns();
          if (!idle_since) idle_since = now;
          if (now - idle_since > kWaitNs) {  // nothing could move for 2 s: give up
            raise_error(a.err, DFLASH_DEV_TIMEOUT);
            bar_seen = 1 << 30;  // treat every barrier as passed and drain
            idle_since = now;
          }
        }
      }
      // never leave with copies in flight
      for (long long i = max(0LL, acount - kPNS); i < acount; ++i)
        mbar_wait(&full[i % kPNS], static_cast<uint32_t>((i / kPNS) & 1));
    }
    return;
  }

  // ================================================================== consumers
  pdl_wait();
  const int g8 = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
  long long i = 0;  // ring position, in step with the producer
  bool ok = true;

  auto arrive = [&]() {
    // generic-proxy writes of this phase become visible to the other CTAs' TMA reads
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    consumer_sync();
    if (tid == 0) atomicAdd(&a.bar[0], 1);
  };

  for (int p = 0; p < a.n_phases; ++p) {
    const PPhase& ph = a.ph[p];
    if (p > 0) grid_wait(&a.bar[0], p * grid, a.err);
    if (ph.type == PH_GEMM) {
      GemmShape g = {};
      g.M = a.M; g.K = ph.K; g.n_tiles = ph.n_tiles; g.ks = ph.ks; g.m_blocks = 1;
      g.paired = ph.paired; g.nseg = ph.nseg; g.units = ph.units;
      for (int s = 0; s < 4; ++s) { g.seg_tile0[s] = ph.seg_tile0[s]; g.seg_rows[s] = ph.seg_rows[s]; }
      g.part = a.part; g.counters = a.counters;
      EpiArgs<bf16> e = {};
      e.M = a.M; e.err = a.err;
      const int l = ph.layer;
      if (ph.epi == EPI_QKV) {
        e.pos = a.pos; e.rope = a.rope; e.max_pos = a.max_pos;
        e.S = a.S; e.hq = a.hq; e.hkv = a.hkv; e.hd = kPHD;
        e.q = a.q; e.kb = a.kb; e.vb = a.vb;
      } else if (ph.epi == EPI_RESID) {
        e.y = a.x; e.ldy = a.d; e.N = a.d;
      } else {
        e.act = a.act; e.F = a.F;
      }
      (void)l;
      long long u0 = ph.units * cta / grid, u1 = ph.units * (cta + 1) / grid;
      long long u = u0;
      float acc[2][2][4];
      while (u < u1) {
        const int t = static_cast<int>(u / ph.ks);
        const int ks0 = static_cast<int>(u % ph.ks);
        const long long tile_end = static_cast<long long>(t + 1) * ph.ks;
        const long long seg_end = min(tile_end, u1);
        const int nk = static_cast<int>(seg_end - u);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int y = 0; y < 2; ++y)
#pragma unroll
            for (int z = 0; z < 4; ++z) acc[x][y][z] = 0.f;
        for (int k = 0; k < nk; ++k, ++i) {
          const int s = static_cast<int>(i % kPNS);
          if (ok && !__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>((i / kPNS) & 1)))) {
            if (lane == 0) raise_error(a.err, DFLASH_DEV_TIMEOUT);
            ok = false;
          }
          if (ok) {
            const uint32_t wbase = smem_u32(stages + s * kPStage);
            const uint32_t abase = wbase + kBM * kBK * 2;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              uint32_t af[2][4], bfr[4];
#pragma unroll
              for (int ms = 0; ms < 2; ++ms)
                ldsm_x4(af[ms], wbase + swz128(warp * 32 + ms * 16 + (mi & 1) * 8 + r8, kk * 2 + (mi >> 1)));
              ldsm_x4(bfr, abase + swz128((mi >> 1) * 8 + r8, kk * 2 + (mi & 1)));
#pragma unroll
              for (int ms = 0; ms < 2; ++ms) {
                mma_bf16(acc[ms][0], af[ms], bfr[0], bfr[1]);
                mma_bf16(acc[ms][1], af[ms], bfr[2], bfr[3]);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
#pragma unroll
        for (int ms = 0; ms < 2; ++ms)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int wr = warp * 32 + ms * 16 + g8, ar = j * 8 + 2 * t4;
            Cs[ar * kPPitch + wr] = acc[ms][j][0];
            Cs[(ar + 1) * kPPitch + wr] = acc[ms][j][1];
            Cs[ar * kPPitch + wr + 8] = acc[ms][j][2];
            Cs[(ar + 1) * kPPitch + wr + 8] = acc[ms][j][3];
          }
        consumer_sync();
        const bool whole = (ks0 == 0) && (seg_end == tile_end);
        bool mine = true;
        if (!whole) {
          const int slot = (u == u0) ? 0 : 1;
          float* dst = a.part + ((long long)cta * 2 + slot) * 16 * kBM;
          for (int x = tid; x < 16 * kBM / 4; x += 128)
            reinterpret_cast<float4*>(dst)[x] =
                *reinterpret_cast<const float4*>(Cs + (x / (kBM / 4)) * kPPitch + (x % (kBM / 4)) * 4);
          const int nc = tile_contributors(ph.units, grid, ph.ks, t, nullptr);
          __threadfence();
          consumer_sync();
          if (tid == 0) {
            const int prev = atomicAdd(&a.counters[t], 1);
            const int last = (prev == nc - 1);
            if (last) { atomicExch(&a.counters[t], 0); __threadfence(); }
            *flag = last;
          }
          consumer_sync();
          mine = *flag != 0;
          if (mine) {
            if (tid == 0) tile_contributors(ph.units, grid, ph.ks, t, cslot);
            consumer_sync();
            for (int x = tid; x < 16 * kBM / 4; x += 128) {
              float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int c0 = 0; c0 < nc; c0 += 4) {
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (c0 + j < nc)
                    v[j] = __ldcg(reinterpret_cast<const float4*>(a.part + (long long)cslot[c0 + j] * 16 * kBM) + x);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  if (c0 + j < nc) { s4.x += v[j].x; s4.y += v[j].y; s4.z += v[j].z; s4.w += v[j].w; }
              }
              *reinterpret_cast<float4*>(Cs + (x / (kBM / 4)) * kPPitch + (x % (kBM / 4)) * 4) = s4;
            }
            consumer_sync();
          }
        }
        if (mine) {
          const int nt = t % ph.n_tiles;
          if (ph.epi == EPI_QKV) tile_epilogue<bf16, EPI_QKV>(Cs, kPPitch, 16, 0, nt, g, e, tid, 128);
          else if (ph.epi == EPI_RESID) tile_epilogue<bf16, EPI_RESID>(Cs, kPPitch, 16, 0, nt, g, e, tid, 128);
          else tile_epilogue<bf16, EPI_SWIGLU>(Cs, kPPitch, 16, 0, nt, g, e, tid, 128);
        }
        consumer_sync();
        u = seg_end;
      }
    } else if (ph.type == PH_ATTN) {
      const int items = a.B * a.hkv * a.nsplit;
      const float sc = 1.4426950408889634f / sqrtf(static_cast<float>(kPHD));
      for (int item = cta; item < items; item += grid) {
        int b, g, p0, p1, np;
        if (!attn_item(a, item, b, g, p0, p1, np)) continue;
        const int T = a.ctx_lens[b];
        if (T < 0 || T > a.max_pages * kPage) {
          if (tid == 0) raise_error(a.err, DFLASH_DEV_BAD_INDEX);
        }
        const int split = (item % (a.hkv * a.nsplit)) % a.nsplit;
        const int qr0 = warp * 16;
        const bf16* qb = a.q + (((long long)b * a.hkv + g) * kPQR + qr0) * kPHD;
        uint32_t qf[kPHD / 16][4];
#pragma unroll
        for (int kk = 0; kk < kPHD / 16; ++kk) {
          qf[kk][0] = *reinterpret_cast<const uint32_t*>(qb + g8 * kPHD + kk * 16 + 2 * t4);
          qf[kk][1] = *reinterpret_cast<const uint32_t*>(qb + (g8 + 8) * kPHD + kk * 16 + 2 * t4);
          qf[kk][2] = *reinterpret_cast<const uint32_t*>(qb + g8 * kPHD + kk * 16 + 8 + 2 * t4);
          qf[kk][3] = *reinterpret_cast<const uint32_t*>(qb + (g8 + 8) * kPHD + kk * 16 + 8 + 2 * t4);
        }
        float o[kPHD / 8][4];
#pragma unroll
        for (int j = 0; j < kPHD / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        for (int pg = p0; pg < p1; ++pg, ++i) {
          const int s = static_cast<int>(i % kPNS);
          if (ok && !__all_sync(0xffffffffu, mbar_wait(&full[s], static_cast<uint32_t>((i / kPNS) & 1)))) {
            if (lane == 0) raise_error(a.err, DFLASH_DEV_TIMEOUT);
            ok = false;
          }
          if (ok) {
            const int valid = (pg < np) ? min(kPage, T - pg * kPage) : a.S;
            const uint32_t kbase = smem_u32(stages + s * kPStage);
            const uint32_t vbase = kbase + 4096;
            float sacc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
            for (int kk = 0; kk < kPHD / 16; ++kk) {
              uint32_t kf[4];
              const int key = (mi >> 1) * 8 + r8, ch = kk * 2 + (mi & 1);
              ldsm_x4(kf, kbase + (ch >> 3) * 2048 + swz128(key, ch & 7));
              mma_bf16(sacc[0], qf[kk], kf[0], kf[1]);
              mma_bf16(sacc[1], qf[kk], kf[2], kf[3]);
            }
#pragma unroll
            for (int nn = 0; nn < 2; ++nn)
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int key = nn * 8 + 2 * t4 + (c & 1);
                sacc[nn][c] = key < valid ? sacc[nn][c] * sc : -INFINITY;
              }
            float mx0 = fmaxf(fmaxf(sacc[0][0], sacc[0][1]), fmaxf(sacc[1][0], sacc[1][1]));
            float mx1 = fmaxf(fmaxf(sacc[0][2], sacc[0][3]), fmaxf(sacc[1][2], sacc[1][3]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float nm0 = fmaxf(m0, mx0), nm1 = fmaxf(m1, mx1);
            const float al0 = exp2f(m0 - nm0), al1 = exp2f(m1 - nm1);
            m0 = nm0;
            m1 = nm1;
            float pp[2][4];
#pragma unroll
            for (int nn = 0; nn < 2; ++nn) {
              pp[nn][0] = exp2f(sacc[nn][0] - nm0);
              pp[nn][1] = exp2f(sacc[nn][1] - nm0);
              pp[nn][2] = exp2f(sacc[nn][2] - nm1);
              pp[nn][3] = exp2f(sacc[nn][3] - nm1);
            }
            l0 = l0 * al0 + pp[0][0] + pp[0][1] + pp[1][0] + pp[1][1];
            l1 = l1 * al1 + pp[0][2] + pp[0][3] + pp[1][2] + pp[1][3];
#pragma unroll
            for (int j = 0; j < kPHD / 8; ++j) {
              o[j][0] *= al0; o[j][1] *= al0;
              o[j][2] *= al1; o[j][3] *= al1;
            }
            uint32_t pa[4], pl[4];
            split_bf16x2(pp[0][0], pp[0][1], pa[0], pl[0]);
            split_bf16x2(pp[0][2], pp[0][3], pa[1], pl[1]);
            split_bf16x2(pp[1][0], pp[1][1], pa[2], pl[2]);
            split_bf16x2(pp[1][2], pp[1][3], pa[3], pl[3]);
#pragma unroll
            for (int dj = 0; dj < kPHD / 16; ++dj) {
              uint32_t vf[4];
              const int key = (mi & 1) * 8 + r8, ch = dj * 2 + (mi >> 1);
              ldsm_x4_trans(vf, vbase + (ch >> 3) * 2048 + swz128(key, ch & 7));
              mma_bf16(o[2 * dj], pa, vf[0], vf[1]);
              mma_bf16(o[2 * dj + 1], pa, vf[2], vf[3]);
              mma_bf16(o[2 * dj], pl, vf[0], vf[1]);
              mma_bf16(o[2 * dj + 1], pl, vf[2], vf[3]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        AttnArgs<bf16> at = {};
        at.S = a.S; at.hq = a.hq; at.hkv = a.hkv; at.hd = kPHD; at.QR = kPQR;
        at.nsplit = a.nsplit; at.part_o = a.part_o; at.out = a.o;
#pragma unroll
        for (int j = 0; j < kPHD / 8; ++j) {
          const int dd = j * 8 + 2 * t4;
          attn_emit<bf16>(at, b, g, split, qr0 + g8, dd, o[j][0], o[j][1], l0);
          attn_emit<bf16>(at, b, g, split, qr0 + g8 + 8, dd, o[j][2], o[j][3], l1);
        }
        if (t4 == 0 && a.nsplit > 1) {
          float* pm = a.part_ml + ((((long long)b * a.hkv + g) * a.nsplit + split) * kPQR + qr0) * 2;
          pm[g8 * 2] = m0;
          pm[g8 * 2 + 1] = l0;
          pm[(g8 + 8) * 2] = m1;
          pm[(g8 + 8) * 2 + 1] = l1;
        }
      }
    } else if (ph.type == PH_COMBINE) {
      // rows (b, g, r) spread over the CTAs; 32 lanes x float4 cover one row of 128
      const int rows = a.B * a.hkv * kPQR;
      for (int row = cta * 4 + warp; row < rows; row += grid * 4) {
        const int b = row / (a.hkv * kPQR), g = (row / kPQR) % a.hkv, r = row % kPQR;
        int T = a.ctx_lens[b];
        if (T < 0 || T > a.max_pages * kPage) T = 0;
        const int ns = ((T + kPage - 1) / kPage + 1 + a.pps - 1) / a.pps;
        const long long grp = (long long)b * a.hkv + g;
        const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + grp * a.nsplit * kPQR;
        const float4* po = reinterpret_cast<const float4*>(a.part_o + grp * a.nsplit * kPQR * kPHD);
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s) M = fmaxf(M, __ldcg(&ml[(long long)s * kPQR + r].x));
        float L = 0.f;
        float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < ns; s0 += 8) {
          float4 v[8];
          float2 qq[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (s0 + j < ns) {
              qq[j] = __ldcg(&ml[(long long)(s0 + j) * kPQR + r]);
              v[j] = __ldcg(&po[((long long)(s0 + j) * kPQR + r) * (kPHD / 4) + lane]);
            }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (s0 + j < ns) {
              const float w = exp2f(qq[j].x - M);
              L += w * qq[j].y;
              acc4.x += w * v[j].x; acc4.y += w * v[j].y; acc4.z += w * v[j].z; acc4.w += w * v[j].w;
            }
        }
        const float inv = 1.f / L;
        const int G = a.hq / a.hkv, ii = r / G, hh = r % G;
        bf16* dst = a.o + ((long long)b * a.S + ii) * a.qw + (g * G + hh) * kPHD + lane * 4;
        dst[0] = from_f32<bf16>(acc4.x * inv);
        dst[1] = from_f32<bf16>(acc4.y * inv);
        dst[2] = from_f32<bf16>(acc4.z * inv);
        dst[3] = from_f32<bf16>(acc4.w * inv);
      }
    } else {  // PH_NORM: row m = cta (rows < grid)
      if (cta < a.M) {
        const bf16* gain = ph.final_norm ? a.g_final
                                         : (ph.epi == 0 ? a.g_mlp[ph.layer] : a.g_attn[ph.layer]);
        bf16* out = ph.final_norm ? a.final_hidden : a.n;
        const float* src = a.x + (long long)cta * a.d;
        float ss = 0.f;
        for (int c = tid * 4; c < a.d; c += 128 * 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + c));
          ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        consumer_sync();
        const float rs = 1.0f / sqrtf((red[0] + red[1] + red[2] + red[3]) / a.d + a.eps);
        for (int c = tid * 4; c < a.d; c += 128 * 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(src + c));
          bf16* o4 = out + (long long)cta * a.d + c;
          o4[0] = from_f32<bf16>(v.x * rs * to_f32<bf16>(gain[c]));
          o4[1] = from_f32<bf16>(v.y * rs * to_f32<bf16>(gain[c + 1]));
          o4[2] = from_f32<bf16>(v.z * rs * to_f32<bf16>(gain[c + 2]));
          o4[3] = from_f32<bf16>(v.w * rs * to_f32<bf16>(gain[c + 3]));
        }
      }
    }
    arrive();
  }
  // all phases done: the last CTA out resets the barrier words for the next launch
  if (tid == 0) {
    const int prev = atomicAdd(&a.bar[1], 1);
    if (prev == grid - 1) {
      atomicExch(&a.bar[0], 0);
      atomicExch(&a.bar[1], 0);
    }
  }
}

#endif  // DFLASH_PERSIST_KERNEL

}  // namespace dflash
