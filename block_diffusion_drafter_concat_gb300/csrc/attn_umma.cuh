// Split-context attention on the 5th-generation tensor cores, for batches of blocks.
//
// One CTA takes one (sequence, kv head, page range) like the mma.sync kernel and
// produces the same online-softmax state, but both contractions run as tcgen05.mma
// with M = 128 query rows (the block's S*G rows of the kv head, padded to 128):
//   S = Q K^T     N = 64 keys (four 16-key pages), K = head_dim;   fp32 in TMEM
//   O += P V      N = head_dim, K = 64 keys, P as a bf16 pair hi + lo (two MMAs)
// Q and the K/V pages arrive by TMA with the 128-byte swizzle (K pages are K-major
// operands, V pages MN-major ones, exactly as they sit in the cache).  P stays in
// tensor memory: the softmax warps write it over the S columns it was computed from
// (hi in the first 32, lo in the last 32) and the P V MMA reads its A operand there.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then four pages of K and V per ring stage
//   warp 1      allocates TMEM (S/P double buffer 2 x 64 columns + O, head_dim
//               columns) and issues the MMAs from one thread: S of step j+1 is
//               computed while the softmax warps work on step j.  MMAs from one thread
//               run in issue order, so S of step j+2 (issued after P V of step j)
//               cannot overwrite P of step j before it has been read.
//   warps 2..5  one query row per thread (TMEM lane): read S, mask, exponentiate
//               against a reference maximum in the log2 domain, write P; O accumulates
//               in TMEM across steps and is rescaled in place only when the reference
//               moves (when a probability could exceed 2^8)
// Key-split mode (at most 64 query rows per kv head, head_dim 64 or 128): the rows are
// loaded twice, into tile rows 0-63 and 64-127; lane r takes keys 0-31 of every step
// and lane r + 64 keys 32-63 of the same query, each with its own reference, row sum
// and O row, and the two states are merged after the last step.
// Every wait is bounded; a role whose wait gives up raises the error word and stops.
#pragma once

#include "attention.cuh"
#include "umma.cuh"

namespace dflash {

// Shared-memory descriptor with explicit leading/stride byte offsets, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128_lbo(uint32_t saddr, uint32_t lbo,
                                                        uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// D (+)= A B with A read from tensor memory (lane = row, two bf16 per column, K along
// the columns) and B from a shared-memory descriptor.
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x by the hardware approximation, subnormal results flushed to zero (the
// probabilities here are relative to a reference at most 2^8 below the row maximum, so
// a flushed value is below 2^-118 of the row's largest term).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Paired fp32 arithmetic (two lanes of a 64-bit register pair per instruction).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Probabilities 2^(x*sc - mref) of N scores in place; returns their sum (four partial
// sums, added pairwise).
template <int N>
__device__ __forceinline__ float exp2_row(float (&x)[N], float sc, float nref) {
  const uint64_t sc2 = f2_pack(sc, sc), nr2 = f2_pack(nref, nref);
  uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int e = 0; e < N / 2; ++e) {
    float t0, t1;
    f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), sc2, nr2), t0, t1);
    x[2 * e] = ex2_ftz(t0);
    x[2 * e + 1] = ex2_ftz(t1);
    const uint64_t pp = f2_pack(x[2 * e], x[2 * e + 1]);
    if (e & 1) acc1 = f2_add(acc1, pp);
    else acc0 = f2_add(acc0, pp);
  }
  float a0, a1, b0, b1;
  f2_unpack(acc0, a0, a1);
  f2_unpack(acc1, b0, b1);
  return (a0 + a1) + (b0 + b1);
}

// Maximum of N values as a tree of three-input maxima.
template <int N>
__device__ __forceinline__ float max_tree(const float (&x)[N]);

// bf16 pair hi = the upper halves of (a, b) (truncation: one byte permute) and the pair
// of residuals lo = bf16(x - hi), rounded to nearest even (x - hi is exact in fp32).
// hi + lo is within 2^-16 of x relative (|x - hi| < 2^-7 |x|, lo's rounding 2^-9 of it).
__device__ __forceinline__ void split_bf16x2_f2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
  hi = __byte_perm(ua, ub, 0x7632);
  float r0, r1;
  f2_unpack(f2_sub(f2_pack(a, b), f2_pack(__uint_as_float(ua & 0xffff0000u),
                                          __uint_as_float(ub & 0xffff0000u))),
            r0, r1);
  lo = pack_bf16x2(r0, r1);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

template <>
__device__ __forceinline__ float max_tree<64>(const float (&x)[64]) {
  float t3[22], u3[8];
#pragma unroll
  for (int i = 0; i < 21; ++i) t3[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  t3[21] = x[63];
#pragma unroll
  for (int i = 0; i < 7; ++i) u3[i] = fmax3(t3[3 * i], t3[3 * i + 1], t3[3 * i + 2]);
  u3[7] = t3[21];
  return fmax3(fmax3(u3[0], u3[1], u3[2]), fmax3(u3[3], u3[4], u3[5]), fmaxf(u3[6], u3[7]));
}

template <>
__device__ __forceinline__ float max_tree<32>(const float (&x)[32]) {
  float t3[11], u3[4];
#pragma unroll
  for (int i = 0; i < 10; ++i) t3[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  t3[10] = fmaxf(x[30], x[31]);
#pragma unroll
  for (int i = 0; i < 3; ++i) u3[i] = fmax3(t3[3 * i], t3[3 * i + 1], t3[3 * i + 2]);
  u3[3] = fmaxf(t3[9], t3[10]);
  return fmax3(u3[0], u3[1], fmaxf(u3[2], u3[3]));
}

template <int HD, bool KSPLIT>
struct AuCfg {
  static constexpr int KT = 64;                    // keys per step
  static constexpr int PG = KT / kPage;            // pages per step
  static constexpr int KB = HD / 64;               // 64-column blocks of a head
  // head_dim 128: one CTA per SM with a five-stage ring (two CTAs would leave room for
  // two 32 KB stages each, one step of lookahead: the loads, not the softmax, bound it)
  static constexpr int CPS = HD == 64 ? 2 : 1;     // CTAs per SM
  static constexpr int NS = 4;                     // ring stages (head_dim 128: 3 and 5 slower)
  static constexpr int NK = KSPLIT ? KT / 2 : KT;  // keys of a step per softmax thread
  static constexpr int Q_BYTES = 128 * HD * 2;
  static constexpr int KV_BLOCK = KT * 128;        // one 64-column block of K or V
  static constexpr int KV_BYTES = KB * KV_BLOCK;
  static constexpr int STAGE = 2 * KV_BYTES;       // K then V
  static constexpr int PAGE_BYTES = kPage * HD * 2;  // one page of K (or V)
  static constexpr int NBAR = 2 * NS + 7;
  static constexpr int SMEM = 1024 + Q_BYTES + NS * STAGE + NBAR * 8 + 16;
  static constexpr int TMEM_COLS = 256;
  static constexpr int O_COL = 2 * KT;             // O: columns [128, 128 + HD)
  static constexpr int THREADS = 192;
  static constexpr uint32_t IDESC_S = umma_idesc_bf16<128, KT>();
  static constexpr uint32_t IDESC_O = umma_idesc_bf16<128, HD>() | (1u << 16);  // B MN-major
  static_assert(O_COL + HD <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  // After the last MMA the K/V ring is idle: the key-split merge buffer (64 rows of O and
  // (m, l)) takes its first half, the staged split output (up to 128 rows x HD fp32, in
  // 32-column slabs) the rest (key-split) or all of it
  static constexpr int STG_OFF = KSPLIT ? NS * STAGE / 2 : 0;
  static constexpr int MAX_QR = KSPLIT ? 64 : 128;
  static_assert(!KSPLIT || 64 * HD * 4 + 2 * 64 * 8 <= STG_OFF, "merge buffer");
  static_assert(STG_OFF + MAX_QR * HD * 4 <= NS * STAGE, "staged output");
  static_assert(32 % PG == 0, "page ids of whole steps per 32 lanes");
};

// Byte pitch of one 32-column slab of the staged output: rows of 128 bytes, whole
// 1024-byte swizzle atoms.
__device__ __forceinline__ int stage_pitch(int QR) { return ((QR + 7) & ~7) * 128; }

// Row `row` of slab `c` (32 fp32 values) into the staged output, 128-byte swizzled as a
// TMA store of a box of 32 columns expects it (eight 16-byte chunks per row, chunk k at
// position k ^ (row & 7): a warp's stores of one chunk hit distinct banks).
__device__ __forceinline__ void stage_row32(uint8_t* stg, int c, int QR, int row,
                                            const uint32_t (&v)[32]) {
  uint8_t* slab = stg + c * stage_pitch(QR);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(slab + swz128(row, k)) =
        make_uint4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

template <int HD, bool KSPLIT>
__global__ void __launch_bounds__(192, AuCfg<HD, KSPLIT>::CPS)
    k_attn_umma(const __grid_constant__ AuMaps maps, const AttnArgs<bf16> a) {
  using C = AuCfg<HD, KSPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sq = smem;                                   // Q: KB blocks of [128][64]
  uint8_t* stages = sq + C::Q_BYTES;                    // K blocks, then V blocks
  uint64_t* kvfull = reinterpret_cast<uint64_t*>(stages + C::NS * C::STAGE);
  uint64_t* kvempty = kvfull + C::NS;
  uint64_t* qfull = kvempty + C::NS;
  uint64_t* sfull = qfull + 1;    // [2] S of a step is in TMEM
  uint64_t* pready = sfull + 2;   // [2] P of a step is in TMEM (over its S)
  uint64_t* ofull = pready + 2;
  uint64_t* done = ofull + 1;
  uint32_t* tbase = reinterpret_cast<uint32_t*>(done + 1);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // context lengths and the page table predate the previous kernel (read before the wait);
  // warp 0 requests the page ids of the split's first 32 pages together with the length
  // (entries past the sequence's pages are read, inside the table's row, but not used)
  int tab0 = 0;
  if (warp == 0 && split * a.pps + lane < a.max_pages)
    tab0 = a.page_table[(long long)b * a.max_pages + split * a.pps + lane];
  const int T = a.ctx_lens[b];
  if (T < 0 || T > a.max_pages * kPage) {
    if (tid == 0) raise_error(a.err, DFLASH_DEV_BAD_INDEX);
    return;
  }
  const int np = (T + kPage - 1) / kPage;   // context pages
  const int kp = np + 1;                    // + the block's own keys
  const int ns = (kp + a.pps - 1) / a.pps;
  if (split >= ns) return;
  const int p0 = split * a.pps, p1 = min(kp, p0 + a.pps);
  const int npg = p1 - p0;
  const int nsteps = (npg + C::PG - 1) / C::PG;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&kvfull[s], 1);
      mbar_init(&kvempty[s], 1);
    }
    mbar_init(qfull, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sfull[k], 1);
      mbar_init(&pready[k], 4);
    }
    mbar_init(ofull, 1);
    mbar_init(done, 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tbase, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    // Q first, after the wait (the previous kernel writes it), then the K/V stages.  A
    // CTA's first S needs Q and the first stage only, and one SM's loads arrive about in
    // the order they were issued at its share of the bandwidth: behind a full ring, Q
    // would come a ring's transfer time later (measured on GB300: Q after the ring
    // 1426 us per Llama-shaped batch-8 step, after the first stage 1397 us, first 1395 us;
    // gpt-oss-shaped batch 64: 4833 / 4796 / 4794 us).
    bool ok = true;
    int issued = 0;
    pdl_wait();
    if (lane == 0) {
      mbar_arrive_expect_tx(qfull, C::Q_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::KB; ++kb) {
        if constexpr (KSPLIT) {
          // the group's (up to) 64 query rows in tile rows 0-63 and again in 64-127
          tma_load_2d(sq + kb * (128 * 128), &maps.q, qfull, kb * 64, (b * a.hkv + g) * a.QR);
          tma_load_2d(sq + kb * (128 * 128) + 64 * 128, &maps.q, qfull, kb * 64,
                      (b * a.hkv + g) * a.QR);
        } else {
          tma_load_2d(sq + kb * (128 * 128), &maps.q, qfull, kb * 64, (b * a.hkv + g) * a.QR);
        }
      }
    }
    // Page ids 32 at a time (SPC steps), lane i holding page 32c + i of the split; the
    // next 32 are requested SPC steps before they are needed, so that the ring's refills
    // never wait on a page-table read.
    constexpr int SPC = 32 / C::PG;
    auto fetch_tab = [&](int j0) {
      const int pg = p0 + j0 * C::PG + lane;
      return (j0 < nsteps && pg < np && pg < p1)
                 ? a.page_table[(long long)b * a.max_pages + pg]
                 : 0;
    };
    int tab = tab0, tab_next = fetch_tab(SPC);
    for (int j = 0; j < nsteps && ok; ++j) {
      const int s = j % C::NS;
      const int pa = j * C::PG;                       // first page of the step in the split
      const int cnt = min(C::PG, npg - pa);
      if (j > 0 && j % SPC == 0) {
        tab = tab_next;
        tab_next = fetch_tab(j + SPC);
      }
      const int tpage = __shfl_sync(0xffffffffu, tab, ((j % SPC) * C::PG + lane) & 31);
      int my_page = 0;
      if (lane < cnt && p0 + pa + lane < np) my_page = tpage;
      if (lane == 0 && j >= C::NS && !mbar_wait(&kvempty[s], ((j / C::NS) - 1) & 1)) {
        raise_error(a.err, DFLASH_DEV_TIMEOUT);
        ok = false;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // Pages past the split's last one are loaded from beyond the pool (zero fill):
      // their scores are masked, but P = 0 must meet finite V rows.
      if (lane == 0) mbar_arrive_expect_tx(&kvfull[s], C::PG * 2 * C::PAGE_BYTES);
      __syncwarp();
      // lane q issues page q's copies (the expected bytes are set above)
      if (lane < C::PG) {
        const int q = lane;
        const int pg = p0 + pa + q;
        const CUtensorMap *mk, *mv;
        int row;
        if (q >= cnt) {
          mk = &maps.k;
          mv = &maps.v;
          row = a.num_pages * a.hkv * kPage;   // first row past the pool
        } else if (pg < np) {
          int page = my_page;
          if (page < 0 || page >= a.num_pages) {
            raise_error(a.err, DFLASH_DEV_BAD_INDEX);
            page = 0;
          }
          mk = &maps.k;
          mv = &maps.v;
          row = (page * a.hkv + g) * kPage;
        } else {
          mk = &maps.kb;
          mv = &maps.vb;
          row = (b * a.hkv + g) * a.S;
        }
        uint8_t* kd = stages + s * C::STAGE + q * (kPage * 128);
        uint8_t* vd = kd + C::KV_BYTES;
#pragma unroll
        for (int kb = 0; kb < C::KB; ++kb) {
          tma_load_2d(kd + kb * C::KV_BLOCK, mk, &kvfull[s], kb * 64, row);
          tma_load_2d(vd + kb * C::KV_BLOCK, mv, &kvfull[s], kb * 64, row);
        }
      }
      issued = j + 1;
    }
    if (lane == 0) {
      // never leave with copies in flight
      mbar_wait(qfull, 0);
      for (int j = max(0, issued - C::NS); j < issued; ++j)
        mbar_wait(&kvfull[j % C::NS], (j / C::NS) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(qfull, 0);
      if (!ok) raise_error(a.err, DFLASH_DEV_TIMEOUT);
      const uint32_t qa = smem_u32(sq);
      auto issue_s = [&](int j) {
        const int s = j % C::NS, sb = j & 1;
        // buffer sb last held P of step j-2, read by the P V MMA issued before this one
        if (!mbar_wait(&kvfull[s], (j / C::NS) & 1)) return false;
        tc_fence_after();
        const uint32_t kbase = smem_u32(stages + s * C::STAGE);
        const uint32_t d = tmem + static_cast<uint32_t>(sb * C::KT);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(qa + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
          const uint64_t bd = umma_desc_sw128(kbase + (kk >> 2) * C::KV_BLOCK + (kk & 3) * 32);
          umma_bf16(d, ad, bd, C::IDESC_S, kk != 0);
        }
        umma_commit(&sfull[sb]);
        return true;
      };
      if (ok && nsteps > 0) ok = issue_s(0);
      for (int j = 0; j < nsteps && ok; ++j) {
        if (j + 1 < nsteps && !issue_s(j + 1)) { ok = false; break; }
        if (!mbar_wait(&pready[j & 1], (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const int s = j % C::NS;
        const uint32_t vbase = smem_u32(stages + s * C::STAGE) + C::KV_BYTES;
        const uint32_t d = tmem + C::O_COL;
        const uint32_t pt = tmem + static_cast<uint32_t>((j & 1) * C::KT);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < C::KT / 16; ++kk) {
            // P: 16 keys = 8 columns of bf16 pairs; hi then lo, 32 columns each
            // V: MN-major (head dims contiguous), 8-key groups 1024 B apart, 64-column
            // blocks of the head KV_BLOCK apart; 16 keys per MMA = two groups
            const uint64_t bd = umma_desc_sw128_lbo(vbase + kk * 2048, C::KV_BLOCK, 1024);
            umma_bf16_ta(d, pt + h * (C::KT / 2) + kk * 8, bd, C::IDESC_O, (j | h | kk) != 0);
          }
        }
        umma_commit(ofull);
        umma_commit(&kvempty[s]);
      }
      if (!ok) raise_error(a.err, DFLASH_DEV_TIMEOUT);
      umma_commit(done);
      mbar_wait(done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warps
    pdl_wait();
    pdl_launch_dependents();
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                     // TMEM lane
    // key split: lanes r and r + 64 hold the same query row; lane r takes keys 0-31 of
    // every step and lane r + 64 keys 32-63, each with its own softmax state and O row,
    // merged after the last step.  Otherwise lane r is query row r with all 64 keys.
    const int half = KSPLIT ? (r >> 6) : 0;
    const int qrow = KSPLIT ? (r & 63) : r;
    constexpr int NK = C::NK;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t o_addr = tmem + lane_base + C::O_COL;
    const float sc = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
    // Reference maximum in the log2 domain: probabilities are 2^(s - mref), O and l
    // accumulate against it (O in TMEM, by the MMAs).  mref moves (to the row max) only
    // when a step's probabilities could exceed 2^8, which stays well inside fp32, so O
    // is rescaled in TMEM rarely; the result does not depend on the reference.
    float mref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nsteps && ok; ++j) {
      const int sb = j & 1;
      const uint32_t s_addr = tmem + lane_base + static_cast<uint32_t>(sb * C::KT);
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[sb], (j >> 1) & 1))) { ok = false; break; }
      tc_fence_after();
      // Raw scores; keys past a page's valid count are masked only in steps that have
      // any (the last steps of a split): the common step is four full pages.  The max is
      // taken on raw scores (the scale is positive) and the scale folded into one FMA
      // with the reference below.
      float x[NK];
      auto load_s = [&]() {
        uint32_t s0[32];
        tmem_ld32(s_addr + half * 32, s0);
        if constexpr (NK == 64) {
          uint32_t s1[32];
          tmem_ld32(s_addr + 32, s1);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) x[32 + k] = __uint_as_float(s1[k]);
        } else {
          tmem_ld_wait();
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(s0[k]);
      };
      load_s();
      int vq[C::PG];
      bool full = true;
#pragma unroll
      for (int q = 0; q < C::PG; ++q) {
        const int pg = p0 + j * C::PG + q;
        vq[q] = pg >= p1 ? 0 : (pg < np) ? min(kPage, T - pg * kPage) : a.S;
        full = full && vq[q] == kPage;
      }
      // Fast path (full steps after the first): exponentiate against the current
      // reference without a row max; the reference only has to move when a probability
      // could exceed 2^8, and a row sum <= 2^8 rules that out.  Otherwise (and on the
      // first step and masked steps) S is read again and the reference moved to the
      // row max.
      float ps = 0.f;
      bool slow = j == 0 || !full;
      bool tried = false;
      if (!slow) {
        tried = true;
        ps = exp2_row<NK>(x, sc, -mref);
        slow = __any_sync(0xffffffffu, !(ps <= 256.f));
      }
      if (slow) {
        if (tried) load_s();
        if (!full) {
          // this thread's keys are pages [q0, q0 + NK / 16) of the step
#pragma unroll
          for (int q = 0; q < NK / kPage; ++q) {
            const int vv = (KSPLIT && half) ? vq[NK / kPage + q] : vq[q];
#pragma unroll
            for (int k = 0; k < kPage; ++k)
              if (k >= vv) x[q * kPage + k] = -INFINITY;
          }
        }
        const float mx = max_tree<NK>(x) * sc;
        const bool move = mx > mref;
        if (__any_sync(0xffffffffu, move)) {
          const float mn = move ? mx : mref;
          const float alpha = exp2f(mref - mn);         // 0 on the first step
          l *= alpha;
          mref = mn;
          if (j > 0) {
            // the previous step's P V must have landed before O is rescaled in place
            if (!__all_sync(0xffffffffu, mbar_wait(ofull, (j - 1) & 1))) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
              uint32_t ov[32];
              tmem_ld32(o_addr + c * 32, ov);
              tmem_ld_wait();
#pragma unroll
              for (int d = 0; d < 32; ++d) ov[d] = __float_as_uint(__uint_as_float(ov[d]) * alpha);
              tmem_st32(o_addr + c * 32, ov);
            }
            tmem_st_wait();
          }
        }
        if (mref == -INFINITY) {
          // no valid key of this thread yet (a key-split half of a one-page split)
#pragma unroll
          for (int k = 0; k < NK; ++k) x[k] = 0.f;
          ps = 0.f;
        } else {
          ps = exp2_row<NK>(x, sc, -mref);
        }
      }
      l += ps;
      // P over this step's S columns: hi pairs in the first 32, lo pairs in the last 32;
      // a key-split thread writes its 16 pairs and zeros for the other half's
      {
        uint32_t hi[32], lo[32];
        if constexpr (NK == 64) {
#pragma unroll
          for (int e = 0; e < 32; ++e) split_bf16x2_f2(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            uint32_t h2, l2;
            split_bf16x2_f2(x[2 * e], x[2 * e + 1], h2, l2);
            hi[e] = half ? 0u : h2;
            hi[16 + e] = half ? h2 : 0u;
            lo[e] = half ? 0u : l2;
            lo[16 + e] = half ? l2 : 0u;
          }
        }
        tmem_st32(s_addr, hi);
        tmem_st32(s_addr + 32, lo);
      }
      tmem_st_wait();
      // Keep the softmax at most one P V ahead: the ofull phases seen by the waits here,
      // in the rescale above and after the loop are then never ambiguous.
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(ofull, (j - 1) & 1))) { ok = false; break; }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[sb]);
    }
    if (ok && nsteps > 0 && !__all_sync(0xffffffffu, mbar_wait(ofull, (nsteps - 1) & 1))) ok = false;
    if (!ok && lane == 0) raise_error(a.err, DFLASH_DEV_TIMEOUT);
    tc_fence_after();
    // split partials (o unnormalised) go out through shared memory and TMA stores of
    // whole 32-column slabs; a single split's normalised output is written directly
    const bool staged = a.nsplit > 1;
    uint8_t* stg = stages + C::STG_OFF;
    if constexpr (KSPLIT) {
      // The K/V ring is idle (every MMA has completed).  Lanes r and r + 64 hold the same
      // query row; each hands the other, through shared memory, the half of its O row
      // that the other merges (lanes 0-63 merge columns [0, HD/2), lanes 64-127 columns
      // [HD/2, HD)), with its (m, l).  Row q's columns are rotated by q so that a warp's
      // 32 stores of one column hit 32 banks.  Both halves form the merged state in the
      // same order (the key-0..31 half's terms first).
      constexpr int HH = HD / 2;
      float* mo = reinterpret_cast<float*>(stages);               // [2][64][HH]
      float* mml = mo + 2 * 64 * HH;                              // [2][64][2]
      float* mine = mo + half * 64 * HH;
      const float* other = mo + (1 - half) * 64 * HH;
      const int give0 = half ? 0 : HH, keep0 = half ? HH : 0;     // columns handed over, kept
#pragma unroll
      for (int c = 0; c < HH / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_addr + give0 + c * 32, ov);
        tmem_ld_wait();
#pragma unroll
        for (int d = 0; d < 32; ++d)
          mine[qrow * HH + ((c * 32 + d + qrow) & (HH - 1))] = __uint_as_float(ov[d]);
      }
      mml[half * 128 + 2 * qrow] = mref;
      mml[half * 128 + 2 * qrow + 1] = l;
      epi_sync();
      const float m2 = mml[(1 - half) * 128 + 2 * qrow], l2 = mml[(1 - half) * 128 + 2 * qrow + 1];
      const float M = fmaxf(mref, m2);
      const float w1 = exp2f(mref - M), w2 = exp2f(m2 - M);
      // (m0, l0, w0): the key-0..31 half's state, whichever thread this is
      const float wa = half ? w2 : w1, wb = half ? w1 : w2;
      l = half ? l2 * wa + l * wb : l * wa + l2 * wb;
      mref = M;
#pragma unroll
      for (int c = 0; c < HH / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_addr + keep0 + c * 32, ov);
        tmem_ld_wait();
        if (qrow < a.QR && ok) {
#pragma unroll
          for (int d = 0; d < 32; ++d) {
            const float own = __uint_as_float(ov[d]);
            const float oth = other[qrow * HH + ((c * 32 + d + qrow) & (HH - 1))];
            ov[d] = __float_as_uint(half ? oth * wa + own * wb : own * wa + oth * wb);
          }
          if (staged) {
            stage_row32(stg, keep0 / 32 + c, a.QR, qrow, ov);
          } else {
#pragma unroll
            for (int d = 0; d < 32; d += 2)
              attn_emit<bf16>(a, b, g, split, qrow, keep0 + c * 32 + d, __uint_as_float(ov[d]),
                              __uint_as_float(ov[d + 1]), l);
          }
        }
      }
    } else {
      // O from TMEM 32 columns at a time (the loads are warp-wide; rows past QR skip the
      // stores only)
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(o_addr + c * 32, ov);
        tmem_ld_wait();
        if (r < a.QR && ok) {
          if (staged) {
            stage_row32(stg, c, a.QR, r, ov);
          } else {
#pragma unroll
            for (int d = 0; d < 32; d += 2)
              attn_emit<bf16>(a, b, g, split, r, c * 32 + d, __uint_as_float(ov[d]),
                              __uint_as_float(ov[d + 1]), l);
          }
        }
      }
    }
    if (staged) {
      fence_proxy_async_smem();
      if (epi_sync_and(ok) && tid == 64) {
        const int y = static_cast<int>((((long long)b * a.hkv + g) * a.nsplit + split) * a.QR);
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) tma_store_2d(&maps.po, stg + c * stage_pitch(a.QR), c * 32, y);
        bulk_commit();
        bulk_wait_read();
      }
    }
    if (!half && qrow < a.QR) {
      if (a.nsplit > 1) {
        const long long grp = (long long)b * a.hkv + g;
        float* pm = a.part_ml + ((grp * a.nsplit + split) * a.QR + qrow) * 2;
        pm[0] = mref;
        pm[1] = l;
      }
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace dflash
