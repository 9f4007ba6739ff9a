// C ABI of libdflash (declared in include/dflash.h): argument validation, workspace
// carving, TMA descriptor encoding and the kernel launch chains of each entry point.
// Every launch carries the programmatic-stream-serialization attribute so that each
// kernel's weight prefetch overlaps the tail of the kernel before it.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <type_traits>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "host.h"
#include "misc.cuh"

using namespace dflash;

// ------------------------------------------------------------------ error plumbing
namespace {
thread_local std::string g_last_error;
thread_local int g_launches = 0;
}  // namespace

namespace dflash {
dflash_status fail(dflash_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}
void count_launch() { ++g_launches; }
}  // namespace dflash

namespace {

#define CUDA_TRY(expr)                                                                   \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess)                                                               \
      return fail(DFLASH_ECUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));         \
  } while (0)

#define TRY(expr) DFLASH_TRY(expr)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// wait limit of the split-tile finishers under the forced-timeout test hook
constexpr unsigned long long kForcedWaitNs = 10000000ull;  // 10 ms

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, inner] with row stride `ld` elements, read in boxes of
// box_rows x 64 elements (128 bytes) with 128-byte swizzle; out-of-range reads give 0.
dflash_status encode_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t inner,
                          uint64_t ld, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled unavailable");
  if (!aligned16(ptr) || (ld * 2) % 16 != 0 || rows == 0 || inner == 0)
    return fail(DFLASH_EINVAL, "tensor %p (%llu x %llu, ld %llu) not TMA-compatible", ptr,
                (unsigned long long)rows, (unsigned long long)inner, (unsigned long long)ld);
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DFLASH_OK;
}

// Row-major fp32 matrix [rows, inner] (row stride inner elements), written by TMA in
// boxes of box_rows x 32 elements (128 bytes) with 128-byte swizzle.
dflash_status encode_f32_store(CUtensorMap* m, void* ptr, uint64_t rows, uint64_t inner,
                               uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled unavailable");
  if (!aligned16(ptr) || (inner * 4) % 16 != 0 || rows == 0 || inner < 32 || box_rows == 0 ||
      box_rows > 256)
    return fail(DFLASH_EINVAL, "fp32 tensor %p (%llu x %llu) not TMA-compatible", ptr,
                (unsigned long long)rows, (unsigned long long)inner);
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled (f32) failed (%d)", (int)r);
  return DFLASH_OK;
}

// Packed FP8 matrix [rows, cols]: e4m3 codes with row stride round_up(cols, 16) bytes,
// then rows fp32 scales at a 256-byte aligned offset.
size_t fp8_ld(long long cols) { return (size_t)((cols + 15) / 16 * 16); }
size_t fp8_scale_offset(long long rows, long long cols) {
  return ((size_t)rows * fp8_ld(cols) + 255) & ~size_t(255);
}
size_t fp8_packed_bytes(long long rows, long long cols) {
  return fp8_scale_offset(rows, cols) + (size_t)rows * sizeof(float);
}

// Codes of a packed FP8 matrix as a byte tensor, read in boxes of box_rows x 128 bytes
// (128 values of k) with 128-byte swizzle; out-of-range reads give 0.
dflash_status encode_fp8(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled unavailable");
  if (!aligned16(ptr) || rows == 0 || cols == 0)
    return fail(DFLASH_EINVAL, "packed FP8 matrix %p (%llu x %llu) not TMA-compatible", ptr,
                (unsigned long long)rows, (unsigned long long)cols);
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {fp8_ld(cols)};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ECUDA, "cuTensorMapEncodeTiled (fp8) failed (%d)", (int)r);
  return DFLASH_OK;
}

// ------------------------------------------------------------------ workspace carving
struct Carve {
  char* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += n * sizeof(T);
    return p;
  }
};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

}  // namespace

// ------------------------------------------------------------------ the handle
struct dflash_handle_s {
  dflash_config c;
  bool bf16;
  int dev = 0, sms = 148;
  const void *w_fuse, *g_fuse, *g_final, *embed, *lm_head;
  std::vector<const void*> g_attn, w_q, w_k, w_v, w_o, g_mlp, w_gate, w_up, w_down;
  CUtensorMap m_fuse, m_lm;
  std::vector<CUtensorMap> m_q, m_k, m_v, m_o, m_gate, m_up, m_down;
  int* d_err = nullptr;
  float2* d_rope = nullptr;
  bool force_timeout = false;  // test hook: split-tile finishers wait for too much
  bool fp8 = false;            // projection weights are packed FP8 (per-row scales)
};

namespace {

using H = dflash_handle_s;

// ------------------------------------------------------------------ GEMM planning
struct WSet {
  const CUtensorMap* maps[kMaxSeg];
  const void* ptrs[kMaxSeg];
  int rows[kMaxSeg];
  int nseg = 0;
  bool paired = false;
  void add(const CUtensorMap* m, const void* p, int r) {
    maps[nseg] = m;
    ptrs[nseg] = p;
    rows[nseg] = r;
    ++nseg;
  }
};

// Activation rows per tile: up to 64 rows the projections stream weights past an
// mma.sync tile; beyond that they are dense contractions for the tcgen05 kernel.
int pick_bn(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

// tcgen05 projections that take whole 256-row tiles run on SM pairs (cta_group::2)
constexpr bool kPairTiles = true;
bool umma_bn(int bn) { return bn >= 128; }

GemmShape plan_shape(const H* h, const WSet& w, int M, int K, bool tc, int* grid_out) {
  GemmShape g = {};
  g.M = M;
  g.K = K;
  g.wait_extra = h->force_timeout ? 1 : 0;
  g.wait_ns = h->force_timeout ? kForcedWaitNs : kWaitNs;
  g.paired = w.paired;
  g.nseg = w.nseg;
  int t = 0;
  for (int s = 0; s < w.nseg; ++s) {
    g.seg_tile0[s] = t;
    g.seg_rows[s] = w.rows[s];
    t += w.paired ? (s == 0 ? ceil_div(w.rows[0], kBM / 2) : 0) : ceil_div(w.rows[s], kBM);
  }
  g.seg_tile0[w.nseg] = t;
  if (w.paired) g.seg_tile0[1] = t;  // both halves of every tile come from segment 0's range
  g.n_tiles = t;
  g.ks = ceil_div(K, h->fp8 ? 2 * kBK : kBK);   // an FP8 stage covers 128 k
  // stream-K: at least 4 units per CTA, and few enough CTAs per tile for the table of
  // the tile's finisher
  const long long per = std::max<long long>(4, (g.ks + 509) / 510);
  const long long ctas = (long long)h->sms * (h->fp8 ? 2 : 1);   // FP8: two CTAs per SM
  auto streamk_grid = [&](long long units) {
    return static_cast<int>(std::min<long long>(ctas, (units + per - 1) / per));
  };
  int bn = tc ? pick_bn(M) : kF32BN;
  if (h->fp8) bn = std::min(bn, 32);   // FP8 weights: the weight-streaming kernel only
  int grid = 0;
  if (tc && umma_bn(bn)) {
    // tcgen05 tiles of 128 or 256 rows, as whole tiles per CTA (waves of tiles) or as
    // stream-K ranges (every SM busy, split tiles finished by their last contributor):
    // the cheaper by a model of times measured on GB300: a k-stage of a 256-row tile
    // ~0.46 us, of a 128-row tile ~0.53 us (both bound by operand delivery, not the
    // MMA), and ~40 us to finish split tiles through the partial buffers.
    constexpr double kStage128 = 0.53, kStage256 = 0.46, kFinish = 40.0;
    double best = 1e30;
    for (int cand : {128, 256}) {
      if (cand == 256 && M <= 128) continue;
      const long long tiles = (long long)ceil_div(M, cand) * g.n_tiles;
      // with many tiles per CTA, stream-K balances to the unit and finishes only a
      // handful of split tiles off the critical path
      const bool many = tiles >= 4LL * h->sms;
      const double st = cand == 256 ? kStage256 : kStage128;
      const long long waves = (tiles + h->sms - 1) / h->sms;
      const double t_tile = (double)waves * g.ks * st;
      const int gs = streamk_grid(tiles * g.ks);
      const bool splits = (tiles * g.ks) % gs != 0 || (tiles * g.ks / gs) % g.ks != 0;
      const double t_sk = (double)((tiles * g.ks + gs - 1) / gs) * st + (splits ? kFinish : 0.0);
      if (!many && t_tile <= best) {
        best = t_tile;
        bn = cand;
        g.tile_mode = 1;
        grid = static_cast<int>((tiles + waves - 1) / waves);
      }
      if (t_sk < best) {
        best = t_sk;
        bn = cand;
        g.tile_mode = 0;
        grid = gs;
      }
    }
  }
  g.bn = bn;
  g.m_blocks = ceil_div(M, bn);
  g.units = (long long)g.m_blocks * g.n_tiles * g.ks;
  if (grid == 0) grid = streamk_grid(g.units);
  if (kPairTiles && tc && bn == 256 && g.tile_mode && !h->fp8) {
    // whole 256-row tiles on SM pairs: a pair takes an activation block against two
    // weight tiles (each SM loads its weight box and half the activation box), in as many
    // waves of pairs as the single-CTA plan had of tiles.  Measured on GB300 (cold, one
    // Qwen3-shaped layer at 512 rows): O 45.3 -> 37 us, Q/K/V and gate/up unchanged (48
    // and 89 us: not bound by operand delivery); graph steps: batch 32 2306 -> 2294 us,
    // gpt-oss batch 64 4775 -> 4751 us.  128-row tiles on pairs were slower (Llama
    // batch 8 1393 -> 1431 us) and stay on single CTAs.
    const long long t2 = (long long)g.m_blocks * ((g.n_tiles + 1) / 2);
    const long long pairs = std::max<long long>(1, h->sms / 2);
    const long long waves = (t2 + pairs - 1) / pairs;
    g.pair = 1;
    grid = static_cast<int>(2 * ((t2 + waves - 1) / waves));
  }
  *grid_out = std::max(1, grid);
  return g;
}

// split-tile partials: two slots per CTA of tiles with up to max_rows activation rows
size_t gemm_part_floats(const H* h, int max_rows) {
  return (size_t)h->sms * (h->fp8 ? 2 : 1) * 2 * pick_bn(std::max(1, max_rows)) * kBM;
}

// Runs one projection: y = A W^T over the weight segments of `w`, epilogue EPI.
template <int EPI, typename T>
dflash_status gemm(const H* h, const void* A, int M, int K, const WSet& w, EpiArgs<T> e,
                   float* part, int* ctr, cudaStream_t st) {
  if (M == 0) return DFLASH_OK;
  int grid;
  const bool tc = h->bf16;
  GemmShape g = plan_shape(h, w, M, K, tc, &grid);
  g.part = part;
  g.counters = ctr;
  e.M = M;
  if (EPI == EPI_F32 || EPI == EPI_RESID || EPI == EPI_ARGMAX || EPI == EPI_ARGKEY)
    e.N = w.rows[0];
  // two control words per tile: arrivals and publications of split pieces
  const int ctl_per_tile = 2;
  if (g.m_blocks * g.n_tiles * ctl_per_tile > 2 * kTileWords)
    return fail(DFLASH_EUNSUPPORTED, "GEMM with %d tiles exceeds the control words",
                g.m_blocks * g.n_tiles);
  if constexpr (std::is_same<T, bf16>::value) {
    CUtensorMap tmA;
    const int bn = g.bn;
    TRY(encode_bf16(&tmA, A, M, K, K, g.pair ? bn / 2 : bn));
    WMaps wm;
    for (int s = 0; s < w.nseg; ++s) wm.m[s] = *w.maps[s];
    if (h->fp8) {
      for (int s = 0; s < w.nseg; ++s)
        g.wscale[s] = reinterpret_cast<const float*>(static_cast<const char*>(w.ptrs[s]) +
                                                     fp8_scale_offset(w.rows[s], K));
      return launch_gemm_tc_f8(bn, EPI, tmA, wm, g, grid, e, st);
    }
    if (umma_bn(bn))
      return g.pair ? launch_gemm_umma_pairs(bn, EPI, tmA, wm, g, grid, e, st)
                    : launch_gemm_umma(bn, EPI, tmA, wm, g, grid, e, st);
    if (bn <= 32) return launch_gemm_tc_lo(bn, EPI, tmA, wm, g, grid, e, st);
    return launch_gemm_tc_hi(bn, EPI, tmA, wm, g, grid, e, st);
  } else {
    WPtrs p = {};
    for (int s = 0; s < w.nseg; ++s) p.p[s] = static_cast<const float*>(w.ptrs[s]);
    return launch_gemm_f32(EPI, dim3(g.m_blocks * g.n_tiles), static_cast<const float*>(A), K, p,
                           g, e, st);
  }
}

// ------------------------------------------------------------------ small launches
template <typename T, typename Tin>
dflash_status rmsnorm(const H* h, const Tin* x, const void* gain, T* y, int rows,
                      cudaStream_t st) {
  if (rows == 0) return DFLASH_OK;
  return launch(k_rmsnorm<T, Tin>, dim3(rows), dim3(kRowThreads), 0, st, x,
                static_cast<float*>(nullptr), static_cast<const T*>(gain), y, h->c.d_model,
                h->c.rms_eps, static_cast<const int*>(nullptr), static_cast<const T*>(nullptr), 0,
                static_cast<const int*>(nullptr), 1, 0, static_cast<int*>(nullptr), h->d_err,
                static_cast<const T*>(nullptr), static_cast<const Tin*>(nullptr),
                static_cast<const T*>(nullptr), 0);
}

// ------------------------------------------------------------------ attention plan
// Blocks of many rows (a batch of sequences) run attention on the tcgen05 kernel: with
// head_dim 64 and up to 128 query rows per kv head one row per TMEM lane, with at most
// 64 rows (head_dim 64 or 128) in key-split mode (each row on two lanes, half of every
// step's keys each).  A single block (latency-bound) stays on the mma.sync kernel.
bool attn_ksplit(const dflash_config& c) {
  return c.block_size * (c.n_q_heads / c.n_kv_heads) <= 64;
}
bool use_attn_umma(const dflash_config& c, int M) {
  const int QR = c.block_size * (c.n_q_heads / c.n_kv_heads);
  if (c.dtype != DFLASH_BF16 || M <= 64) return false;
  return (c.head_dim == 64 && QR <= 128) || (c.head_dim == 128 && QR <= 64);
}

struct AttnPlan {
  int pps, nsplit;
};

AttnPlan plan_attn(const H* h, int B, int max_pages, bool causal = false) {
  const int kp = max_pages + 1;
  const long long groups = (long long)B * h->c.n_kv_heads;
  if (use_attn_umma(h->c, B * h->c.block_size) && !causal) {
    // tcgen05 kernel (two CTAs per SM at head_dim 64, one at 128), four pages per step:
    // whole steps per split and the fewest waves of CTAs times steps per CTA (plus about
    // three steps of per-CTA prologue and epilogue); among plans within 2 % of the best,
    // the fewest splits.
    const long long slots = (h->c.head_dim == 64 ? 2LL : 1LL) * h->sms;
    AttnPlan best{0, 0};
    long long best_cost = 0;
    for (int ns = 1; ns <= std::min(64, ceil_div(kp, 4)); ++ns) {
      const int pps = ceil_div(ceil_div(kp, ns), 4) * 4;
      const int nsr = ceil_div(kp, pps);
      if (nsr != ns) continue;
      const long long cost = (groups * ns + slots - 1) / slots * (pps / 4 + 3);
      if (best.nsplit == 0 || cost * 50 < best_cost * 49) {
        best = {pps, ns};
        best_cost = cost;
      }
    }
    // Key-split mode (head_dim 128, steps bound by K/V bandwidth): the model assumes
    // every sequence has the longest context.  When it leaves one CTA more than 40
    // steps, a batch of ragged lengths would wait on its longest sequence's few CTAs,
    // so splits of 24 steps are taken instead (measured on GB300: ragged batch 32
    // 2604 -> 2498 us per step; a uniform batch 8 keeps its 33-step plan).
    if (attn_ksplit(h->c) && best.pps / 4 > 40) {
      const int pps = std::max(96, ceil_div(ceil_div(kp, 64), 4) * 4);   // <= 64 splits
      best = {pps, ceil_div(kp, pps)};
    }
    return best;
  }
  // mma.sync kernel: about eight (b, kv head, split) CTAs per SM at the longest context,
  // so that ragged lengths and the last wave of CTAs balance; at least kMinPages pages
  // (each CTA's pages are one chain of dependent steps; fewer splits mean a longer chain,
  // more a bigger combine: measured on GB300 at batch 1, context 2048, 6 pages per split
  // beat 4 by 4.6 us a step and 8 by 4.5 us) and at most 64 splits.
  constexpr int kMinPages = 6;
  const long long want = std::max<long long>(1, (8LL * h->sms + groups - 1) / groups);
  const long long cap = std::min(64, ceil_div(kp, kMinPages));
  const int ns = static_cast<int>(std::min(want, cap));
  const int pps = std::max(kMinPages, ceil_div(kp, ns));
  return {pps, ceil_div(kp, pps)};
}

// ------------------------------------------------------------------ workspace plans
// rows of a block plus new context rows that one weight-streaming tile takes
constexpr int kInjRows = 64;

struct DraftWs {
  int* ctl;
  float* x;
  void* n;
  int* pos;
  void *q, *kb, *vb, *o, *act;
  float *part_o, *part_ml, *gpart;
  float* u;   // fusion projection of merged-injection rows (fp32)
};

size_t elt(const H* h) { return h->bf16 ? 2 : 4; }

DraftWs carve_draft(const H* h, Carve& cv, int B, int max_pages) {
  const auto& c = h->c;
  const size_t M = (size_t)B * c.block_size;
  // split partials for the larger of the block's plan and a causal chunk's plan
  const AttnPlan pb = plan_attn(h, B, max_pages), pc = plan_attn(h, B, max_pages, true);
  const AttnPlan ap = pb.nsplit >= pc.nsplit ? pb : pc;
  const int QR = c.block_size * (c.n_q_heads / c.n_kv_heads);
  DraftWs w;
  w.ctl = cv.take<int>(kCtlWords);
  w.x = cv.take<float>(M * c.d_model);
  // normed rows, then room for up to kInjRows fused context rows that a merged
  // injection appends to the Q/K/V projection's activations
  w.n = cv.take<char>((M + kInjRows) * c.d_model * elt(h));
  w.pos = cv.take<int>(M);
  w.q = cv.take<char>(M * c.n_q_heads * c.head_dim * elt(h));
  w.kb = cv.take<char>((M + 16) * c.n_kv_heads * c.head_dim * elt(h));
  w.vb = cv.take<char>((M + 16) * c.n_kv_heads * c.head_dim * elt(h));
  w.o = cv.take<char>(M * c.n_q_heads * c.head_dim * elt(h));
  w.act = cv.take<char>(M * c.ffn_dim * elt(h));
  w.part_o = cv.take<float>((size_t)B * c.n_kv_heads * ap.nsplit * QR * c.head_dim);
  w.part_ml = cv.take<float>((size_t)B * c.n_kv_heads * ap.nsplit * QR * 2);
  w.gpart = cv.take<float>(gemm_part_floats(h, std::max(static_cast<int>(M), kInjRows)));
  w.u = cv.take<float>((size_t)kInjRows * c.d_model);
  return w;
}

// a causal chunk of context rows for the input-fusion drafter: the block's buffers plus
// the fusion's fp32 projection and its normed rows
struct InputsWs {
  DraftWs d;
  float* u;
  void* fused;
};

InputsWs carve_inputs(const H* h, Carve& cv, int B, int max_pages) {
  InputsWs w;
  w.d = carve_draft(h, cv, B, max_pages);
  const size_t M = (size_t)B * h->c.block_size;
  w.u = cv.take<float>(M * h->c.d_model);
  w.fused = cv.take<char>(M * h->c.d_model * elt(h));
  return w;
}

// a target chunk: the block's buffers plus the final hidden rows of the LM head
struct TargetWs {
  DraftWs d;
  void* hfin;
};

TargetWs carve_target(const H* h, Carve& cv, int B, int max_pages) {
  TargetWs w;
  w.d = carve_draft(h, cv, B, max_pages);
  w.hfin = cv.take<char>((size_t)B * h->c.block_size * h->c.d_model * elt(h));
  return w;
}

struct InjectWs {
  int* ctl;
  float* u;
  void* fused;
  float* gpart;
};

InjectWs carve_inject(const H* h, Carve& cv, int n) {
  InjectWs w;
  w.ctl = cv.take<int>(kCtlWords);
  w.u = cv.take<float>((size_t)n * h->c.d_model);
  w.fused = cv.take<char>((size_t)n * h->c.d_model * elt(h));
  w.gpart = cv.take<float>(gemm_part_floats(h, n));
  return w;
}

struct HeadWs {
  int* ctl;
  float *am_max, *am_sum;
  int* am_idx;
  float* gpart;
};

HeadWs carve_head(const H* h, Carve& cv, int rows) {
  const size_t t = (size_t)ceil_div(h->c.vocab, kBM) * rows;
  HeadWs w;
  w.ctl = cv.take<int>(kCtlWords);
  w.am_max = cv.take<float>(t);
  w.am_sum = cv.take<float>(t);
  w.am_idx = cv.take<int>(t);
  w.gpart = cv.take<float>(gemm_part_floats(h, rows));
  return w;
}

int verify_chunks(const H* h, int rows) {
  const int V = h->c.vocab;
  int nch = std::max(1, ceil_div(2 * h->sms, rows));
  int chunk = std::max(2048, ceil_div(ceil_div(V, nch), 2048) * 2048);
  return ceil_div(V, chunk);
}
int chunk_of(const H* h, int nch) {
  int c = ceil_div(h->c.vocab, nch);
  return ceil_div(c, 8) * 8;
}

struct VerifyWs {
  int* ctl;
  float *pv, *pv2, *lse_t, *zr;
  int* pi;
  int* rej;
  void* hrow;
  float* gpart;
};

VerifyWs carve_verify(const H* h, Carve& cv, int B, bool sample) {
  const int rows = B * h->c.block_size;
  const int nch = verify_chunks(h, rows);
  VerifyWs w = {};
  w.ctl = cv.take<int>(kCtlWords);
  w.pv = cv.take<float>((size_t)rows * nch);
  w.pv2 = cv.take<float>((size_t)rows * nch);
  w.pi = cv.take<int>((size_t)rows * nch);
  if (sample) {
    w.lse_t = cv.take<float>(rows);
    w.rej = cv.take<int>(B);
    w.hrow = cv.take<char>((size_t)B * h->c.d_model * elt(h));
    w.zr = cv.take<float>((size_t)B * h->c.vocab);
    w.gpart = cv.take<float>(gemm_part_floats(h, B));
  }
  return w;
}

dflash_status check_ws(const void* ws, size_t have, size_t need) {
  if (!ws) return fail(DFLASH_EINVAL, "workspace is NULL");
  if (!aligned16(ws)) return fail(DFLASH_EINVAL, "workspace not 16-byte aligned");
  if (have < need)
    return fail(DFLASH_EWORKSPACE, "workspace %zu bytes < %zu needed", have, need);
  return DFLASH_OK;
}

// Every call on a handle enqueues work for the handle's device: that device must be the
// current one (kernels, workspace and the device scratch array all live there).
dflash_status check_device(const dflash_handle_s* h) {
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev != h->dev)
    return fail(DFLASH_EINVAL, "the handle belongs to device %d but device %d is current",
                h->dev, dev);
  return DFLASH_OK;
}

#define CHECK_HANDLE(h)                                                                  \
  do {                                                                                   \
    if (!(h)) return fail(DFLASH_EINVAL, "null handle");                                 \
    TRY(check_device(h));                                                                \
  } while (0)

#define NEED(p, what)                                                                    \
  do {                                                                                   \
    if (!(p)) return fail(DFLASH_EINVAL, "%s is NULL", what);                            \
    if (!aligned16(p)) return fail(DFLASH_EINVAL, "%s not 16-byte aligned", what);       \
  } while (0)

}  // namespace

// fused = RMSNorm(x_cat W_fuse^T) with gain g_fuse (norm = false: only u = x_cat W_fuse^T)
static dflash_status fuse_impl(H* h, const void* x_cat, int n, void* fused, float* u,
                               float* gpart, int* ctl, cudaStream_t st, bool norm = true) {
  const int kin = h->c.n_target_layers * h->c.target_width;
  WSet w;
  w.add(&h->m_fuse, h->w_fuse, h->c.d_model);
  if (h->bf16) {
    EpiArgs<bf16> e = {};
    e.y = u;
    e.ldy = h->c.d_model;
    e.err = h->d_err;
    TRY((gemm<EPI_F32, bf16>(h, x_cat, n, kin, w, e, gpart, ctl, st)));
    if (!norm) return DFLASH_OK;
    return rmsnorm<bf16, float>(h, u, h->g_fuse, static_cast<bf16*>(fused), n, st);
  }
  EpiArgs<float> e = {};
  e.y = u;
  e.ldy = h->c.d_model;
  e.err = h->d_err;
  TRY((gemm<EPI_F32, float>(h, x_cat, n, kin, w, e, gpart, ctl, st)));
  if (!norm) return DFLASH_OK;
  return rmsnorm<float, float>(h, u, h->g_fuse, static_cast<float*>(fused), n, st);
}

static dflash_status inject_impl(H* h, const void* f, int n, const int32_t* positions,
                                 const int32_t* slots, int32_t num_pages, void* const* k_pool,
                                 void* const* v_pool, const InjectWs& w, cudaStream_t st) {
  const auto& c = h->c;
  // one GEMM per group of up to 8 layers: segments k_l | v_l
  for (int l0 = 0; l0 < c.n_layers; l0 += kMaxSeg / 2) {
    const int nl = std::min(kMaxSeg / 2, c.n_layers - l0);
    WSet ws_;
    for (int l = l0; l < l0 + nl; ++l) {
      ws_.add(h->bf16 ? &h->m_k[l] : nullptr, h->w_k[l], c.n_kv_heads * c.head_dim);
      ws_.add(h->bf16 ? &h->m_v[l] : nullptr, h->w_v[l], c.n_kv_heads * c.head_dim);
    }
    auto fill = [&](auto& e, auto* tag) {
      using T = std::remove_pointer_t<decltype(tag)>;
      e.pos = positions;
      e.rope = h->d_rope;
      e.max_pos = c.max_position;
      e.S = c.block_size;
      e.hq = c.n_q_heads;
      e.hkv = c.n_kv_heads;
      e.hd = c.head_dim;
      for (int l = 0; l < nl; ++l) {
        e.kpool[l] = static_cast<T*>(k_pool[l0 + l]);
        e.vpool[l] = static_cast<T*>(v_pool[l0 + l]);
      }
      e.slots = slots;
      e.num_slots = (long long)num_pages * kPage;
      e.err = h->d_err;
    };
    if (h->bf16) {
      EpiArgs<bf16> e = {};
      fill(e, static_cast<bf16*>(nullptr));
      TRY((gemm<EPI_KV, bf16>(h, f, n, c.d_model, ws_, e, w.gpart, w.ctl, st)));
    } else {
      EpiArgs<float> e = {};
      fill(e, static_cast<float*>(nullptr));
      TRY((gemm<EPI_KV, float>(h, f, n, c.d_model, ws_, e, w.gpart, w.ctl, st)));
    }
  }
  return DFLASH_OK;
}

// One pass of the layer stack over S rows per sequence at positions ctx_lens[b] + i.
// The drafter's block: token ids in, every row sees all S block keys, final norm out.
// A causal chunk (context rows of the input-fusion drafter, target tokens): input rows
// or ids, row i sees block keys 0..i, each layer's K/V of the rows go into the cache,
// optional taps of the residual stream after given layers.
struct StackOpts {
  const int32_t* ids = nullptr;   // [B, S] token ids (embedding input), or
  const void* rows = nullptr;     // [B*S, d] input rows
  bool causal = false;
  bool write_cache = false;
  const int32_t* tap_layers = nullptr;  // host array, 1-based layer indices
  int n_taps = 0;
  void* taps = nullptr;           // [B*S, n_taps*d]
  void* final_hidden = nullptr;   // [B*S, d] final RMSNorm output, or nullptr
  // merged injection: n_inj fused context rows (in the workspace after the block's
  // normed rows) whose K/V every layer's Q/K/V projection writes to the cache
  int n_inj = 0;
  const int32_t* inj_pos = nullptr;
  const int32_t* inj_slots = nullptr;
  // the fused rows before their RMSNorm (fp32): normalised by the step's first launch
  // together with the block's embedding rows
  const float* inj_u = nullptr;
};

template <typename T>
static dflash_status draft_impl(H* h, const StackOpts& o, const int32_t* ctx_lens,
                                const int32_t* page_table, int32_t max_pages, int32_t B,
                                int32_t num_pages, void* const* k_pool, void* const* v_pool,
                                const DraftWs& w, cudaStream_t st) {
  const auto& c = h->c;
  const int S = c.block_size, M = B * S, d = c.d_model;
  const int qw = c.n_q_heads * c.head_dim, kvw = c.n_kv_heads * c.head_dim;
  const int G = c.n_q_heads / c.n_kv_heads, QR = S * G;
  T* n = static_cast<T*>(w.n);
  // embedding (or input rows) + first pre-attention norm + positions (and the fused
  // context rows' norm, rows M.. of the same launch)
  const int n_u = o.inj_u ? o.n_inj : 0;
  TRY(launch(k_rmsnorm<T, float>, dim3(M + n_u), dim3(kRowThreads), 0, st,
             static_cast<const float*>(nullptr), w.x, static_cast<const T*>(h->g_attn[0]), n, d,
             c.rms_eps, o.ids, static_cast<const T*>(h->embed), c.vocab, ctx_lens, S,
             c.max_position, w.pos, h->d_err, static_cast<const T*>(o.rows), o.inj_u,
             static_cast<const T*>(h->g_fuse), M));
  const AttnPlan ap = plan_attn(h, B, max_pages, o.causal);
  // a chunk whose only output is the cache needs no attention or MLP in its last layer
  const bool kv_only_last = o.write_cache && !o.final_hidden && o.n_taps == 0;
  for (int l = 0; l < c.n_layers; ++l) {
    {  // Q, K, V with RoPE
      WSet ws_;
      ws_.add(h->bf16 ? &h->m_q[l] : nullptr, h->w_q[l], qw);
      ws_.add(h->bf16 ? &h->m_k[l] : nullptr, h->w_k[l], kvw);
      ws_.add(h->bf16 ? &h->m_v[l] : nullptr, h->w_v[l], kvw);
      EpiArgs<T> e = {};
      e.pos = w.pos;
      e.rope = h->d_rope;
      e.max_pos = c.max_position;
      e.S = S;
      e.hq = c.n_q_heads;
      e.hkv = c.n_kv_heads;
      e.hd = c.head_dim;
      e.q = static_cast<T*>(w.q);
      e.kb = static_cast<T*>(w.kb);
      e.vb = static_cast<T*>(w.vb);
      e.err = h->d_err;
      if (o.n_inj) {   // + the new context rows: K/V into this layer's pages
        e.n_inj = o.n_inj;
        e.inj_pos = o.inj_pos;
        e.inj_slots = o.inj_slots;
        e.inj_kpool = static_cast<T*>(k_pool[l]);
        e.inj_vpool = static_cast<T*>(v_pool[l]);
        e.num_slots = (long long)num_pages * kPage;
      }
      TRY((gemm<EPI_QKV, T>(h, n, M + o.n_inj, d, ws_, e, w.gpart, w.ctl, st)));
    }
    if (o.write_cache)
      TRY(launch(k_chunk_kv_to_cache<T>, dim3(M), dim3(kRowThreads), 0, st,
                 static_cast<const T*>(w.kb), static_cast<const T*>(w.vb), ctx_lens, page_table,
                 max_pages, num_pages, static_cast<T*>(k_pool[l]), static_cast<T*>(v_pool[l]), S,
                 c.n_kv_heads, c.head_dim, h->d_err));
    if (kv_only_last && l + 1 == c.n_layers) break;
    {  // attention over [context pages ; block]
      AttnArgs<T> a = {};
      a.q = static_cast<const T*>(w.q);
      a.kb = static_cast<const T*>(w.kb);
      a.vb = static_cast<const T*>(w.vb);
      a.kpool = static_cast<const T*>(k_pool[l]);
      a.vpool = static_cast<const T*>(v_pool[l]);
      a.page_table = page_table;
      a.max_pages = max_pages;
      a.ctx_lens = ctx_lens;
      a.num_pages = num_pages;
      a.S = S;
      a.hq = c.n_q_heads;
      a.hkv = c.n_kv_heads;
      a.hd = c.head_dim;
      a.QR = QR;
      a.pps = ap.pps;
      a.nsplit = ap.nsplit;
      a.part_o = w.part_o;
      a.part_ml = w.part_ml;
      a.out = static_cast<T*>(w.o);
      a.err = h->d_err;
      a.causal = o.causal ? 1 : 0;
      a.fresh = o.n_inj;   // the injected rows are the sequences' newest positions
      dim3 grid(ap.nsplit, c.n_kv_heads, B);
      if constexpr (std::is_same<T, bf16>::value) {
        AttnMaps mp;
        const uint64_t pool_rows = (uint64_t)num_pages * c.n_kv_heads * kPage;
        TRY(encode_bf16(&mp.k, k_pool[l], pool_rows, c.head_dim, c.head_dim, kPage));
        TRY(encode_bf16(&mp.v, v_pool[l], pool_rows, c.head_dim, c.head_dim, kPage));
        const uint64_t blk_rows = (uint64_t)B * c.n_kv_heads * S;
        TRY(encode_bf16(&mp.kb, w.kb, blk_rows, c.head_dim, c.head_dim, kPage));
        TRY(encode_bf16(&mp.vb, w.vb, blk_rows, c.head_dim, c.head_dim, kPage));
        if (use_attn_umma(c, M) && !o.causal) {
          AuMaps am = {};
          am.k = mp.k;
          am.v = mp.v;
          am.kb = mp.kb;
          am.vb = mp.vb;
          const bool ks = attn_ksplit(c);
          TRY(encode_bf16(&am.q, w.q, (uint64_t)B * c.n_kv_heads * QR, c.head_dim, c.head_dim,
                          ks ? 64 : 128));
          // split partials of O leave the kernel as TMA stores of QR x 32 boxes
          if (ap.nsplit > 1)
            TRY(encode_f32_store(&am.po, w.part_o, (uint64_t)B * c.n_kv_heads * ap.nsplit * QR,
                                 c.head_dim, QR));
          TRY(launch_attn_umma(c.head_dim, ks, grid, am, a, st));
        } else {
          TRY(launch_attn_tc(c.head_dim, QR / 16, grid, attn_tc_smem(c.head_dim), mp, a, st));
        }
      } else {
        const int smem = (2 * QR * c.head_dim + 2 * kPage * c.head_dim + QR * kPage + 3 * QR) * 4;
        TRY(launch_attn_f32(grid, smem, a, st));
      }
      if (ap.nsplit > 1) TRY(launch_attn_combine(B, a, st));
    }
    {  // output projection + residual
      WSet ws_;
      ws_.add(h->bf16 ? &h->m_o[l] : nullptr, h->w_o[l], d);
      EpiArgs<T> e = {};
      e.y = w.x;
      e.ldy = d;
      e.err = h->d_err;
      TRY((gemm<EPI_RESID, T>(h, w.o, M, qw, ws_, e, w.gpart, w.ctl, st)));
    }
    TRY((rmsnorm<T, float>(h, w.x, h->g_mlp[l], n, M, st)));
    {  // gate | up with SwiGLU
      WSet ws_;
      ws_.add(h->bf16 ? &h->m_gate[l] : nullptr, h->w_gate[l], c.ffn_dim);
      ws_.add(h->bf16 ? &h->m_up[l] : nullptr, h->w_up[l], c.ffn_dim);
      ws_.paired = true;
      EpiArgs<T> e = {};
      e.act = static_cast<T*>(w.act);
      e.F = c.ffn_dim;
      e.err = h->d_err;
      TRY((gemm<EPI_SWIGLU, T>(h, n, M, d, ws_, e, w.gpart, w.ctl, st)));
    }
    {  // down projection + residual
      WSet ws_;
      ws_.add(h->bf16 ? &h->m_down[l] : nullptr, h->w_down[l], d);
      EpiArgs<T> e = {};
      e.y = w.x;
      e.ldy = d;
      e.err = h->d_err;
      TRY((gemm<EPI_RESID, T>(h, w.act, M, c.ffn_dim, ws_, e, w.gpart, w.ctl, st)));
    }
    for (int t = 0; t < o.n_taps; ++t)
      if (o.tap_layers[t] == l + 1)
        TRY(launch(k_tap<T>, dim3(M), dim3(kRowThreads), 0, st, static_cast<const float*>(w.x),
                   d, static_cast<T*>(o.taps), o.n_taps * d, t * d));
    if (l + 1 < c.n_layers)
      TRY((rmsnorm<T, float>(h, w.x, h->g_attn[l + 1], n, M, st)));
    else if (o.final_hidden)
      TRY((rmsnorm<T, float>(h, w.x, h->g_final, static_cast<T*>(o.final_hidden), M, st)));
  }
  return DFLASH_OK;
}

template <typename T>
static dflash_status head_impl(H* h, const void* hidden, int rows, float temperature,
                               int32_t* tokens, float* max_logit, float* lse, const HeadWs& w,
                               cudaStream_t st) {
  WSet ws_;
  ws_.add(h->bf16 ? &h->m_lm : nullptr, h->lm_head, h->c.vocab);
  EpiArgs<T> e = {};
  e.am_max = w.am_max;
  e.am_idx = w.am_idx;
  e.am_sum = w.am_sum;
  e.inv_temp = 1.0f / temperature;
  e.want_sum = lse != nullptr;
  e.err = h->d_err;
  if (!lse && rows <= 128 && h->bf16) {
    // greedy, one or a few blocks: the argmax is finished inside the projection (packed
    // keys, last CTA).  With more rows the per-row atomics contend (every n-tile hits
    // every row's key), so tile partials and a reduction launch are used instead.
    e.am_key = reinterpret_cast<unsigned long long*>(w.ctl + kKeyWord);
    e.am_done = w.ctl + kDoneWord;
    e.tok_out = tokens;
    e.max_out = max_logit;
    return gemm<EPI_ARGKEY, T>(h, hidden, rows, h->c.d_model, ws_, e, w.gpart, w.ctl, st);
  }
  TRY((gemm<EPI_ARGMAX, T>(h, hidden, rows, h->c.d_model, ws_, e, w.gpart, w.ctl, st)));
  const int n_tiles = ceil_div(h->c.vocab, kBM);
  return launch(k_argmax_finalize, dim3(ceil_div(rows, kRowThreads / 32)), dim3(kRowThreads), 0,
                st, static_cast<const float*>(w.am_max), static_cast<const int*>(w.am_idx),
                static_cast<const float*>(w.am_sum), n_tiles, rows, 1.0f / temperature, tokens,
                max_logit, lse);
}

template <typename T>
static dflash_status sample_impl(H* h, const int32_t* draft, const void* final_hidden,
                                 const float* dmax, const float* dlse, const void* logits,
                                 const float* u, float temperature, int B, int32_t* out_tokens,
                                 int32_t* n_acc, int32_t* n_emit, const VerifyWs& w,
                                 cudaStream_t st) {
  const int S = h->c.block_size, V = h->c.vocab, d = h->c.d_model, rows = B * S;
  const float it = 1.0f / temperature;
  const int nch = verify_chunks(h, rows), chunk = chunk_of(h, nch);
  TRY(launch(k_verify_sample_accept<T>, dim3(nch, rows), dim3(kRowThreads), 0, st,
             static_cast<const T*>(logits), draft, dmax, dlse, u,
             static_cast<const T*>(final_hidden), d, S, V, chunk, it, w.pv, w.pv2, w.lse_t, w.ctl,
             w.rej, static_cast<T*>(w.hrow), out_tokens, n_acc, n_emit, h->d_err));
  {  // drafter logits of each sequence's first rejected slot
    WSet ws_;
    ws_.add(h->bf16 ? &h->m_lm : nullptr, h->lm_head, V);
    EpiArgs<T> e = {};
    e.y = w.zr;
    e.ldy = V;
    e.err = h->d_err;
    TRY((gemm<EPI_F32, T>(h, w.hrow, B, d, ws_, e, w.gpart, w.ctl, st)));
  }
  const int nch2 = verify_chunks(h, B), chunk2 = chunk_of(h, nch2);
  return launch(k_verify_sample_residual<T>, dim3(nch2, B), dim3(kRowThreads), 0, st,
                static_cast<const T*>(logits), static_cast<const float*>(w.zr),
                static_cast<const float*>(w.lse_t), dlse, u, static_cast<const int*>(w.rej), S, V,
                chunk2, it, w.pv, w.pv2, w.ctl, out_tokens);
}

// ===================================================================== entry points
extern "C" {

const char* dflash_last_error(void) { return g_last_error.c_str(); }
int32_t dflash_last_launch_count(void) { return g_launches; }

dflash_status dflash_create(const dflash_config* cfg, const dflash_weights* w,
                            dflash_handle* out) {
  g_launches = 0;
  if (!cfg || !w || !out) return fail(DFLASH_EINVAL, "null argument");
  *out = nullptr;
  const dflash_config& c = *cfg;
  if (c.d_model <= 0 || c.n_layers <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 ||
      c.head_dim <= 0 || c.ffn_dim <= 0 || c.vocab <= 0 || c.block_size <= 0 ||
      c.n_target_layers <= 0 || c.target_width <= 0 || c.max_position <= 0)
    return fail(DFLASH_EINVAL, "non-positive dimension in config");
  if (c.page_size != kPage) return fail(DFLASH_EUNSUPPORTED, "page_size must be 16");
  if (c.n_q_heads % c.n_kv_heads) return fail(DFLASH_EINVAL, "n_q_heads %% n_kv_heads != 0");
  if (c.head_dim % 2) return fail(DFLASH_EINVAL, "head_dim must be even");
  // the rotary pairs of a head are finished inside one 128-column projection tile
  if (kBM % c.head_dim) return fail(DFLASH_EUNSUPPORTED, "head_dim must divide 128");
  if (!(c.rope_theta > 0.f) || !(c.rms_eps >= 0.f)) return fail(DFLASH_EINVAL, "bad theta/eps");
  if (c.dtype != DFLASH_BF16 && c.dtype != DFLASH_F32) return fail(DFLASH_EINVAL, "bad dtype");
  if (c.weight_format != DFLASH_WEIGHTS_NATIVE && c.weight_format != DFLASH_WEIGHTS_FP8)
    return fail(DFLASH_EINVAL, "bad weight_format %d", c.weight_format);
  if (c.weight_format == DFLASH_WEIGHTS_FP8 && c.dtype != DFLASH_BF16)
    return fail(DFLASH_EUNSUPPORTED, "FP8 weights need the bf16 dtype");
  const int QR = c.block_size * (c.n_q_heads / c.n_kv_heads);
  const int kin = c.n_target_layers * c.target_width;
  if (c.dtype == DFLASH_BF16) {
    if (c.head_dim != 64 && c.head_dim != 128)
      return fail(DFLASH_EUNSUPPORTED, "bf16 kernels need head_dim 64 or 128");
    if ((c.n_q_heads * c.head_dim) % kBM || (c.n_kv_heads * c.head_dim) % kBM)
      return fail(DFLASH_EUNSUPPORTED, "q and kv widths must be multiples of 128");
    if (c.d_model % 8 || c.ffn_dim % 8 || kin % 8)
      return fail(DFLASH_EUNSUPPORTED, "widths must be multiples of 8");
    if (QR % 16 || QR > 128 || c.block_size > 16)
      return fail(DFLASH_EUNSUPPORTED, "block_size*group must be a multiple of 16 <= 128");
  } else {
    if (QR > 128 || c.head_dim > 128 || c.block_size > 16)
      return fail(DFLASH_EUNSUPPORTED, "fp32 path: block*group <= 128, head_dim <= 128");
  }
  const void* const* arrs[] = {w->g_attn, w->w_q, w->w_k, w->w_v, w->w_o,
                               w->g_mlp, w->w_gate, w->w_up, w->w_down};
  for (auto a : arrs)
    if (!a) return fail(DFLASH_EINVAL, "per-layer weight array is NULL");
  const void* singles[] = {w->g_final, w->embed, w->lm_head};
  for (auto p : singles) NEED(p, "weight");
  // a handle without fusion weights is a plain transformer (e.g. a target model)
  if ((w->w_fuse == nullptr) != (w->g_fuse == nullptr))
    return fail(DFLASH_EINVAL, "w_fuse and g_fuse must both be given or both be NULL");
  if (w->w_fuse) {
    NEED(w->w_fuse, "w_fuse");
    NEED(w->g_fuse, "g_fuse");
  }
  for (auto a : arrs)
    for (int l = 0; l < c.n_layers; ++l) NEED(a[l], "layer weight");

  H* h = new H();
  h->c = c;
  h->bf16 = c.dtype == DFLASH_BF16;
  h->fp8 = c.weight_format == DFLASH_WEIGHTS_FP8;
  cudaGetDevice(&h->dev);
  cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->dev);
  h->w_fuse = w->w_fuse; h->g_fuse = w->g_fuse; h->g_final = w->g_final;
  h->embed = w->embed; h->lm_head = w->lm_head;
  auto cp = [&](std::vector<const void*>& v, const void* const* a) { v.assign(a, a + c.n_layers); };
  cp(h->g_attn, w->g_attn); cp(h->w_q, w->w_q); cp(h->w_k, w->w_k); cp(h->w_v, w->w_v);
  cp(h->w_o, w->w_o); cp(h->g_mlp, w->g_mlp); cp(h->w_gate, w->w_gate); cp(h->w_up, w->w_up);
  cp(h->w_down, w->w_down);

  auto bail = [&](dflash_status s) {
    if (h->d_err) cudaFree(h->d_err);
    if (h->d_rope) cudaFree(h->d_rope);
    delete h;
    return s;
  };
  if (h->bf16) {
    const int d = c.d_model, qw = c.n_q_heads * c.head_dim, kvw = c.n_kv_heads * c.head_dim;
    // a weight matrix [rows, cols] as TMA boxes of box_rows rows: bf16, or packed FP8
    auto enc = [&](CUtensorMap* m, const void* p, int rows, int cols, int box_rows) {
      return h->fp8 ? encode_fp8(m, p, rows, cols, box_rows)
                    : encode_bf16(m, p, rows, cols, cols, box_rows);
    };
    dflash_status s = h->w_fuse ? enc(&h->m_fuse, h->w_fuse, d, kin, kBM) : DFLASH_OK;
    if (s == DFLASH_OK) s = enc(&h->m_lm, h->lm_head, c.vocab, d, kBM);
    h->m_q.resize(c.n_layers); h->m_k.resize(c.n_layers); h->m_v.resize(c.n_layers);
    h->m_o.resize(c.n_layers); h->m_gate.resize(c.n_layers); h->m_up.resize(c.n_layers);
    h->m_down.resize(c.n_layers);
    for (int l = 0; l < c.n_layers && s == DFLASH_OK; ++l) {
      s = enc(&h->m_q[l], h->w_q[l], qw, d, kBM);
      if (s == DFLASH_OK) s = enc(&h->m_k[l], h->w_k[l], kvw, d, kBM);
      if (s == DFLASH_OK) s = enc(&h->m_v[l], h->w_v[l], kvw, d, kBM);
      if (s == DFLASH_OK) s = enc(&h->m_o[l], h->w_o[l], d, qw, kBM);
      if (s == DFLASH_OK) s = enc(&h->m_gate[l], h->w_gate[l], c.ffn_dim, d, kBM / 2);
      if (s == DFLASH_OK) s = enc(&h->m_up[l], h->w_up[l], c.ffn_dim, d, kBM / 2);
      if (s == DFLASH_OK) s = enc(&h->m_down[l], h->w_down[l], d, c.ffn_dim, kBM);
    }
    if (s != DFLASH_OK) return bail(s);
  }
  if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess ||
      cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess)
    return bail(fail(DFLASH_ECUDA, "cannot allocate the error word"));
  // RoPE table: angle p * theta^(-2j/hd) in double, stored as fp32 (cos, sin)
  const int half = c.head_dim / 2;
  std::vector<float2> tab((size_t)c.max_position * half);
  for (int p = 0; p < c.max_position; ++p)
    for (int j = 0; j < half; ++j) {
      double ang = p * std::pow((double)c.rope_theta, -2.0 * j / c.head_dim);
      tab[(size_t)p * half + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  if (cudaMalloc(&h->d_rope, tab.size() * sizeof(float2)) != cudaSuccess ||
      cudaMemcpy(h->d_rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
          cudaSuccess)
    return bail(fail(DFLASH_ECUDA, "cannot allocate the RoPE table"));
  *out = h;
  return DFLASH_OK;
}

dflash_status dflash_destroy(dflash_handle h) {
  if (!h) return fail(DFLASH_EINVAL, "null handle");
  cudaFree(h->d_err);
  cudaFree(h->d_rope);
  delete h;
  return DFLASH_OK;
}

dflash_status dflash_workspace_size(dflash_handle h, int32_t max_rows, int32_t max_batch,
                                    int32_t max_pages, size_t* bytes) {
  if (!h || !bytes) return fail(DFLASH_EINVAL, "null argument");
  if (max_rows < 0 || max_batch < 0 || max_pages < 0) return fail(DFLASH_EINVAL, "negative size");
  size_t need = 0;
  {
    Carve cv{nullptr};
    carve_inject(h, cv, std::max(max_rows, 1));
    need = std::max(need, cv.off);
  }
  {
    Carve cv{nullptr};
    carve_draft(h, cv, std::max(max_batch, 1), std::max(max_pages, 1));
    need = std::max(need, cv.off);
  }
  {
    Carve cv{nullptr};
    carve_head(h, cv, std::max(max_rows, 1));
    need = std::max(need, cv.off);
  }
  {
    Carve cv{nullptr};
    carve_inputs(h, cv, std::max(max_batch, 1), std::max(max_pages, 1));
    need = std::max(need, cv.off);
  }
  {
    Carve cv{nullptr};
    carve_target(h, cv, std::max(max_batch, 1), std::max(max_pages, 1));
    need = std::max(need, cv.off);
  }
  {
    Carve cv{nullptr};
    carve_verify(h, cv, std::max(max_batch, 1), true);
    need = std::max(need, cv.off);
  }
  *bytes = need;
  return DFLASH_OK;
}

dflash_status dflash_workspace_init(dflash_handle h, void* ws, size_t ws_bytes, void* stream) {
  CHECK_HANDLE(h);
  TRY(check_ws(ws, ws_bytes, kCtlWords * sizeof(int)));
  CUDA_TRY(cudaMemsetAsync(ws, 0, kCtlWords * sizeof(int), static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

dflash_status dflash_fuse_features(dflash_handle h, const void* x_cat, int32_t n, void* fused,
                                   void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (n < 0) return fail(DFLASH_EINVAL, "n < 0");
  if (n == 0) return DFLASH_OK;
  if (!h->w_fuse) return fail(DFLASH_EINVAL, "the handle has no fusion weights");
  NEED(x_cat, "x_cat");
  NEED(fused, "fused");
  Carve cv{static_cast<char*>(ws)};
  InjectWs w = carve_inject(h, cv, n);
  TRY(check_ws(ws, ws_bytes, cv.off));
  return fuse_impl(h, x_cat, n, fused, w.u, w.gpart, w.ctl, static_cast<cudaStream_t>(stream));
}

dflash_status dflash_inject_kv(dflash_handle h, const void* x_cat, const void* fused, int32_t n,
                               const int32_t* positions, const int32_t* slots, int32_t num_pages,
                               void* const* k_pool, void* const* v_pool, void* fused_out,
                               void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (n < 0 || num_pages <= 0) return fail(DFLASH_EINVAL, "bad n or num_pages");
  if (n == 0) return DFLASH_OK;
  if ((x_cat == nullptr) == (fused == nullptr))
    return fail(DFLASH_EINVAL, "exactly one of x_cat and fused must be given");
  if (x_cat) NEED(x_cat, "x_cat");
  if (x_cat && !h->w_fuse) return fail(DFLASH_EINVAL, "the handle has no fusion weights");
  if (fused) NEED(fused, "fused");
  if (fused_out) NEED(fused_out, "fused_out");
  NEED(positions, "positions");
  NEED(slots, "slots");
  if (!k_pool || !v_pool) return fail(DFLASH_EINVAL, "pool arrays are NULL");
  for (int l = 0; l < h->c.n_layers; ++l) {
    NEED(k_pool[l], "k_pool[l]");
    NEED(v_pool[l], "v_pool[l]");
  }
  Carve cv{static_cast<char*>(ws)};
  InjectWs w = carve_inject(h, cv, n);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* f = fused;
  if (x_cat) {
    void* dst = fused_out ? fused_out : w.fused;
    TRY(fuse_impl(h, x_cat, n, dst, w.u, w.gpart, w.ctl, st));
    f = dst;
  }
  return inject_impl(h, f, n, positions, slots, num_pages, k_pool, v_pool, w, st);
}

}  // extern "C"

namespace {
// Host checks shared by the calls that run the layer stack over S rows per sequence.
dflash_status check_stack_args(const H* h, const int32_t* ctx_lens, const int32_t* page_table,
                               int32_t max_pages, int32_t batch, int32_t num_pages,
                               void* const* k_pool, void* const* v_pool) {
  if (batch < 0 || max_pages < 0 || num_pages <= 0) return fail(DFLASH_EINVAL, "bad sizes");
  NEED(ctx_lens, "ctx_lens");
  if (max_pages > 0) NEED(page_table, "page_table");
  if (!k_pool || !v_pool) return fail(DFLASH_EINVAL, "pool arrays are NULL");
  for (int l = 0; l < h->c.n_layers; ++l) {
    NEED(k_pool[l], "k_pool[l]");
    NEED(v_pool[l], "v_pool[l]");
  }
  if ((long long)batch * h->c.block_size > (1 << 20) ||
      (long long)batch * h->c.n_kv_heads > 2 * kTileWords)
    return fail(DFLASH_EUNSUPPORTED, "batch too large");
  return DFLASH_OK;
}
}  // namespace

extern "C" {

dflash_status dflash_draft_block(dflash_handle h, const int32_t* block_ids,
                                 const int32_t* ctx_lens, const int32_t* page_table,
                                 int32_t max_pages, int32_t batch, int32_t num_pages,
                                 void* const* k_pool, void* const* v_pool, void* final_hidden,
                                 void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (batch < 0 || max_pages < 0 || num_pages <= 0) return fail(DFLASH_EINVAL, "bad sizes");
  if (batch == 0) return DFLASH_OK;
  NEED(block_ids, "block_ids");
  NEED(ctx_lens, "ctx_lens");
  if (max_pages > 0) NEED(page_table, "page_table");
  NEED(final_hidden, "final_hidden");
  if (!k_pool || !v_pool) return fail(DFLASH_EINVAL, "pool arrays are NULL");
  for (int l = 0; l < h->c.n_layers; ++l) {
    NEED(k_pool[l], "k_pool[l]");
    NEED(v_pool[l], "v_pool[l]");
  }
  if ((long long)batch * h->c.block_size > (1 << 20)) return fail(DFLASH_EUNSUPPORTED, "batch too large");
  Carve cv{static_cast<char*>(ws)};
  DraftWs w = carve_draft(h, cv, batch, max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  if ((long long)batch * h->c.n_kv_heads > 2 * kTileWords) return fail(DFLASH_EUNSUPPORTED, "batch too large");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StackOpts o;
  o.ids = block_ids;
  o.final_hidden = final_hidden;
  if (h->bf16)
    return draft_impl<bf16>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool,
                            v_pool, w, st);
  return draft_impl<float>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool,
                           v_pool, w, st);
}

dflash_status dflash_inject_draft(dflash_handle h, const void* x_cat, int32_t n_inj,
                                  const int32_t* positions, const int32_t* slots,
                                  const int32_t* block_ids, const int32_t* ctx_lens,
                                  const int32_t* page_table, int32_t max_pages, int32_t batch,
                                  int32_t num_pages, void* const* k_pool, void* const* v_pool,
                                  void* fused_out, void* final_hidden, void* ws, size_t ws_bytes,
                                  void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  const auto& c = h->c;
  const long long M = (long long)batch * c.block_size;
  // one weight-streaming tile holds the block and the new rows, and the attention is
  // the mma.sync kernel (which fetches the fresh pages after its wait)
  const bool merged = h->bf16 && batch > 0 && n_inj > 0 && M + n_inj <= kInjRows &&
                      !use_attn_umma(c, static_cast<int>(M));
  if (!merged) {
    int total = 0;
    TRY(dflash_inject_kv(h, x_cat, nullptr, n_inj, positions, slots, num_pages, k_pool, v_pool,
                         fused_out, ws, ws_bytes, stream));
    total += g_launches;
    TRY(dflash_draft_block(h, block_ids, ctx_lens, page_table, max_pages, batch, num_pages,
                           k_pool, v_pool, final_hidden, ws, ws_bytes, stream));
    g_launches += total;
    return DFLASH_OK;
  }
  if (!h->w_fuse) return fail(DFLASH_EINVAL, "the handle has no fusion weights");
  NEED(x_cat, "x_cat");
  NEED(positions, "positions");
  NEED(slots, "slots");
  NEED(block_ids, "block_ids");
  NEED(final_hidden, "final_hidden");
  if (fused_out) NEED(fused_out, "fused_out");
  TRY(check_stack_args(h, ctx_lens, page_table, max_pages, batch, num_pages, k_pool, v_pool));
  Carve cv{static_cast<char*>(ws)};
  DraftWs w = carve_draft(h, cv, batch, max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // fused rows straight after the block's normed rows: the Q/K/V projections read both
  char* rows = static_cast<char*>(w.n) + (size_t)M * c.d_model * elt(h);
  TRY(fuse_impl(h, x_cat, n_inj, rows, w.u, w.gpart, w.ctl, st, false));
  StackOpts o;
  o.ids = block_ids;
  o.final_hidden = final_hidden;
  o.n_inj = n_inj;
  o.inj_pos = positions;
  o.inj_slots = slots;
  o.inj_u = w.u;
  TRY(draft_impl<bf16>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool, v_pool,
                       w, st));
  // the fused rows stay where the first launch normalised them (no later launch writes
  // them)
  if (fused_out)
    CUDA_TRY(cudaMemcpyAsync(fused_out, rows, (size_t)n_inj * c.d_model * elt(h),
                             cudaMemcpyDeviceToDevice, st));
  return DFLASH_OK;
}



dflash_status dflash_inject_inputs(dflash_handle h, const void* x_cat, const int32_t* ctx_lens,
                                   const int32_t* page_table, int32_t max_pages, int32_t batch,
                                   int32_t num_pages, void* const* k_pool, void* const* v_pool,
                                   void* fused_out, void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  TRY(check_stack_args(h, ctx_lens, page_table, max_pages, batch, num_pages, k_pool, v_pool));
  if (batch == 0) return DFLASH_OK;
  if (!h->w_fuse) return fail(DFLASH_EINVAL, "the handle has no fusion weights");
  NEED(x_cat, "x_cat");
  if (fused_out) NEED(fused_out, "fused_out");
  Carve cv{static_cast<char*>(ws)};
  InputsWs w = carve_inputs(h, cv, batch, max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int M = batch * h->c.block_size;
  void* fused = fused_out ? fused_out : w.fused;
  TRY(fuse_impl(h, x_cat, M, fused, w.u, w.d.gpart, w.d.ctl, st));
  StackOpts o;
  o.rows = fused;
  o.causal = true;
  o.write_cache = true;
  if (h->bf16)
    return draft_impl<bf16>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool,
                            v_pool, w.d, st);
  return draft_impl<float>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool,
                           v_pool, w.d, st);
}

dflash_status dflash_target_forward(dflash_handle h, const int32_t* ids, const int32_t* ctx_lens,
                                    const int32_t* page_table, int32_t max_pages, int32_t batch,
                                    int32_t num_pages, void* const* k_pool, void* const* v_pool,
                                    const int32_t* tap_layers, int32_t n_taps, void* taps,
                                    float* logits, void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  TRY(check_stack_args(h, ctx_lens, page_table, max_pages, batch, num_pages, k_pool, v_pool));
  if (batch == 0) return DFLASH_OK;
  NEED(ids, "ids");
  if (n_taps < 0 || (n_taps > 0 && (!tap_layers || !taps)))
    return fail(DFLASH_EINVAL, "taps: n_taps %d with tap_layers %p, taps %p", n_taps,
                (const void*)tap_layers, taps);
  if (taps) NEED(taps, "taps");
  for (int t = 0; t < n_taps; ++t)
    if (tap_layers[t] < 1 || tap_layers[t] > h->c.n_layers)
      return fail(DFLASH_EINVAL, "tap layer %d outside 1..%d", tap_layers[t], h->c.n_layers);
  if (logits) NEED(logits, "logits");
  Carve cv{static_cast<char*>(ws)};
  TargetWs w = carve_target(h, cv, batch, max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StackOpts o;
  o.ids = ids;
  o.causal = true;
  o.write_cache = true;
  o.tap_layers = tap_layers;
  o.n_taps = n_taps;
  o.taps = taps;
  o.final_hidden = logits ? w.hfin : nullptr;
  const int M = batch * h->c.block_size;
  if (h->bf16) {
    TRY(draft_impl<bf16>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool, v_pool,
                         w.d, st));
  } else {
    TRY(draft_impl<float>(h, o, ctx_lens, page_table, max_pages, batch, num_pages, k_pool,
                          v_pool, w.d, st));
  }
  if (!logits) return DFLASH_OK;
  // the target's logits of every row, fp32 (verification reads them)
  WSet ws_;
  ws_.add(h->bf16 ? &h->m_lm : nullptr, h->lm_head, h->c.vocab);
  if (h->bf16) {
    EpiArgs<bf16> e = {};
    e.y = logits;
    e.ldy = h->c.vocab;
    e.err = h->d_err;
    return gemm<EPI_F32, bf16>(h, w.hfin, M, h->c.d_model, ws_, e, w.d.gpart, w.d.ctl, st);
  }
  EpiArgs<float> e = {};
  e.y = logits;
  e.ldy = h->c.vocab;
  e.err = h->d_err;
  return gemm<EPI_F32, float>(h, w.hfin, M, h->c.d_model, ws_, e, w.d.gpart, w.d.ctl, st);
}

}  // extern "C"

// ------------------------------------------------------------------ speculative loop
namespace {
// The loop's workspace: a region for the drafter's calls (block pass, LM head,
// verification scratch, injection; they run one after another), a region for the
// target's block pass, then the buffers that live from one call of the step to the next.
struct SpecWs {
  char* dreg;
  char* treg;
  void *hidden, *taps;
  int *draft, *tids, *out, *nacc, *pos, *slots;
  float *logits, *dmax;
  size_t dreg_bytes, treg_bytes;
};

size_t region_bytes(const H* hd, int B, int max_pages) {
  const int M = B * hd->c.block_size;
  size_t need = 0;
  auto upd = [&](auto f) {
    Carve cv{nullptr};
    f(cv);
    need = std::max(need, cv.off);
  };
  upd([&](Carve& cv) { carve_draft(hd, cv, B, max_pages); });
  upd([&](Carve& cv) { carve_head(hd, cv, M); });
  upd([&](Carve& cv) { carve_inject(hd, cv, M); });
  upd([&](Carve& cv) { carve_verify(hd, cv, B, false); });
  return (need + 255) & ~size_t(255);
}

SpecWs carve_spec(const H* hd, const H* ht, Carve& cv, int B, int max_pages) {
  const int M = B * hd->c.block_size;
  SpecWs w;
  w.dreg_bytes = region_bytes(hd, B, max_pages);
  Carve ct{nullptr};
  carve_target(ht, ct, B, max_pages);
  w.treg_bytes = (ct.off + 255) & ~size_t(255);
  w.dreg = cv.take<char>(w.dreg_bytes);
  w.treg = cv.take<char>(w.treg_bytes);
  w.hidden = cv.take<char>((size_t)M * hd->c.d_model * elt(hd));
  w.taps = cv.take<char>((size_t)M * hd->c.n_target_layers * hd->c.target_width * elt(hd));
  w.draft = cv.take<int>(M);
  w.tids = cv.take<int>(M);
  w.out = cv.take<int>(M);
  w.nacc = cv.take<int>(B);
  w.pos = cv.take<int>(M);
  w.slots = cv.take<int>(M);
  w.logits = cv.take<float>((size_t)M * ht->c.vocab);
  w.dmax = cv.take<float>(M);
  return w;
}

dflash_status check_pair(const H* hd, const H* ht) {
  const auto &a = hd->c, &b = ht->c;
  if (!hd->w_fuse) return fail(DFLASH_EINVAL, "the drafter handle has no fusion weights");
  if (b.d_model != a.target_width || b.vocab != a.vocab || b.block_size != a.block_size ||
      b.dtype != a.dtype || hd->dev != ht->dev)
    return fail(DFLASH_EINVAL,
                "target (d %d, vocab %d, block %d) does not match the drafter (target width "
                "%d, vocab %d, block %d), or dtype/device differ",
                b.d_model, b.vocab, b.block_size, a.target_width, a.vocab, a.block_size);
  return DFLASH_OK;
}

template <typename T>
dflash_status spec_impl(H* hd, H* ht, const dflash_spec_state& s, const SpecWs& w,
                        cudaStream_t st) {
  const int B = s.batch, S = hd->c.block_size, M = B * S, V = hd->c.vocab;
  int* draft = s.drafts ? s.drafts : w.draft;
  // 1. draft the block [anchor, mask, ...] over the drafter's cache
  {
    Carve cv{w.dreg};
    DraftWs dw = carve_draft(hd, cv, B, s.max_pages);
    StackOpts o;
    o.ids = s.block_ids;
    o.final_hidden = w.hidden;
    TRY(draft_impl<T>(hd, o, s.ctx_lens, s.page_table, s.max_pages, B, s.num_pages, s.d_k_pool,
                      s.d_v_pool, dw, st));
  }
  // 2. the drafter's tokens (LM head + argmax, logits never stored)
  {
    Carve cv{w.dreg};
    HeadWs hw = carve_head(hd, cv, M);
    TRY(head_impl<T>(hd, w.hidden, M, 1.0f, draft, w.dmax, nullptr, hw, st));
  }
  // 3. the target's pass over [anchor, drafts 1..S-1]: its cache, the tap features of
  //    the block's tokens and fp32 logits of every row
  TRY(launch(k_spec_target_ids, dim3(ceil_div(M, 128)), dim3(128), 0, st,
             static_cast<const int*>(s.block_ids), static_cast<const int*>(draft), M, S,
             w.tids));
  {
    Carve cv{w.treg};
    TargetWs tw = carve_target(ht, cv, B, s.max_pages);
    StackOpts o;
    o.ids = w.tids;
    o.causal = true;
    o.write_cache = true;
    o.tap_layers = s.tap_layers;
    o.n_taps = hd->c.n_target_layers;
    o.taps = w.taps;
    o.final_hidden = tw.hfin;
    TRY(draft_impl<T>(ht, o, s.ctx_lens, s.page_table, s.max_pages, B, s.num_pages, s.t_k_pool,
                      s.t_v_pool, tw.d, st));
    WSet ws_;
    ws_.add(ht->bf16 ? &ht->m_lm : nullptr, ht->lm_head, V);
    EpiArgs<T> e = {};
    e.y = w.logits;
    e.ldy = V;
    e.err = ht->d_err;
    TRY((gemm<EPI_F32, T>(ht, tw.hfin, M, ht->c.d_model, ws_, e, tw.d.gpart, tw.d.ctl, st)));
  }
  // 4. synthetic agreement (optional), then greedy verification with the anchor in slot 0
  if (s.plant_u)
    TRY(launch(k_spec_plant, dim3(M), dim3(kRowThreads), 0, st, w.logits,
               static_cast<const int*>(draft), s.plant_u, s.plant_steps,
               static_cast<const int*>(s.step), s.plant_p, S, V, M, hd->d_err));
  {
    Carve cv{w.dreg};
    VerifyWs vw = carve_verify(hd, cv, B, false);
    const int nch = verify_chunks(hd, M), chunk = chunk_of(hd, nch);
    TRY(launch(k_verify_greedy<float>, dim3(nch, M), dim3(kRowThreads), 0, st,
               static_cast<const float*>(w.logits), static_cast<const int*>(draft), S, V,
               chunk, vw.pv, vw.pi, vw.ctl, w.out, w.nacc, s.n_emitted, hd->d_err, 1));
  }
  // 5. commit: emitted tokens, next anchor, context length, injection slots
  TRY(launch(k_spec_commit, dim3(ceil_div(B, 64)), dim3(64), 0, st,
             static_cast<const int*>(w.out), static_cast<const int*>(s.n_emitted), B, S,
             s.mask_id, s.block_ids, s.ctx_lens, s.page_table, s.max_pages, w.pos, w.slots,
             s.generated, s.max_new, s.n_generated, s.step, hd->d_err));
  // 6. the block's target features into the drafter's cache (every row: rows past the
  //    new context length are overwritten by the next step's injection)
  {
    Carve cv{w.dreg};
    InjectWs iw = carve_inject(hd, cv, M);
    TRY(fuse_impl(hd, w.taps, M, iw.fused, iw.u, iw.gpart, iw.ctl, st));
    TRY(inject_impl(hd, iw.fused, M, w.pos, w.slots, s.num_pages, s.d_k_pool, s.d_v_pool, iw,
                    st));
  }
  return DFLASH_OK;
}
}  // namespace

extern "C" {

dflash_status dflash_spec_workspace_size(dflash_handle drafter, dflash_handle target,
                                         int32_t batch, int32_t max_pages, size_t* bytes) {
  if (!drafter || !target || !bytes) return fail(DFLASH_EINVAL, "null argument");
  if (batch <= 0 || max_pages <= 0) return fail(DFLASH_EINVAL, "bad sizes");
  TRY(check_pair(drafter, target));
  Carve cv{nullptr};
  carve_spec(drafter, target, cv, batch, max_pages);
  *bytes = cv.off;
  return DFLASH_OK;
}

dflash_status dflash_spec_workspace_init(dflash_handle drafter, dflash_handle target,
                                         int32_t batch, int32_t max_pages, void* ws,
                                         size_t ws_bytes, void* stream) {
  CHECK_HANDLE(drafter);
  CHECK_HANDLE(target);
  TRY(check_pair(drafter, target));
  Carve cv{static_cast<char*>(ws)};
  SpecWs w = carve_spec(drafter, target, cv, batch, max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemsetAsync(w.dreg, 0, kCtlWords * sizeof(int), st));
  CUDA_TRY(cudaMemsetAsync(w.treg, 0, kCtlWords * sizeof(int), st));
  return DFLASH_OK;
}

dflash_status dflash_spec_step(dflash_handle drafter, dflash_handle target,
                               const dflash_spec_state* s, void* ws, size_t ws_bytes,
                               void* stream) {
  g_launches = 0;
  CHECK_HANDLE(drafter);
  CHECK_HANDLE(target);
  if (!s) return fail(DFLASH_EINVAL, "null state");
  TRY(check_pair(drafter, target));
  if (s->batch <= 0) return fail(DFLASH_EINVAL, "batch must be positive");
  TRY(check_stack_args(drafter, s->ctx_lens, s->page_table, s->max_pages, s->batch,
                       s->num_pages, s->d_k_pool, s->d_v_pool));
  TRY(check_stack_args(target, s->ctx_lens, s->page_table, s->max_pages, s->batch,
                       s->num_pages, s->t_k_pool, s->t_v_pool));
  NEED(s->block_ids, "block_ids");
  NEED(s->generated, "generated");
  NEED(s->n_generated, "n_generated");
  NEED(s->n_emitted, "n_emitted");
  NEED(s->step, "step");
  if (s->drafts) NEED(s->drafts, "drafts");
  if (!s->tap_layers) return fail(DFLASH_EINVAL, "tap_layers is NULL");
  for (int t = 0; t < drafter->c.n_target_layers; ++t)
    if (s->tap_layers[t] < 1 || s->tap_layers[t] > target->c.n_layers)
      return fail(DFLASH_EINVAL, "tap layer %d outside 1..%d", s->tap_layers[t],
                  target->c.n_layers);
  if (s->max_new <= 0) return fail(DFLASH_EINVAL, "max_new must be positive");
  if (s->mask_id < 0 || s->mask_id >= drafter->c.vocab) return fail(DFLASH_EINVAL, "bad mask_id");
  if (s->plant_u) {
    NEED(s->plant_u, "plant_u");
    if (s->plant_steps <= 0) return fail(DFLASH_EINVAL, "plant_steps must be positive");
  }
  if (drafter->c.block_size < 2) return fail(DFLASH_EUNSUPPORTED, "block_size must be >= 2");
  const long long M = (long long)s->batch * drafter->c.block_size;
  if (M > 65535) return fail(DFLASH_EUNSUPPORTED, "batch*block_size > 65535");
  Carve cv{static_cast<char*>(ws)};
  SpecWs w = carve_spec(drafter, target, cv, s->batch, s->max_pages);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (drafter->bf16) return spec_impl<bf16>(drafter, target, *s, w, st);
  return spec_impl<float>(drafter, target, *s, w, st);
}

dflash_status dflash_lm_head_argmax(dflash_handle h, const void* hidden, int32_t rows,
                                    float temperature, int32_t* tokens, float* max_logit,
                                    float* lse, void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (rows < 0) return fail(DFLASH_EINVAL, "rows < 0");
  if (rows == 0) return DFLASH_OK;
  NEED(hidden, "hidden");
  NEED(tokens, "tokens");
  if (max_logit) NEED(max_logit, "max_logit");
  if (lse) NEED(lse, "lse");
  if (lse && !(temperature > 0.f)) return fail(DFLASH_EINVAL, "temperature must be > 0");
  if (!(temperature > 0.f)) temperature = 1.0f;
  Carve cv{static_cast<char*>(ws)};
  HeadWs w = carve_head(h, cv, rows);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->bf16) return head_impl<bf16>(h, hidden, rows, temperature, tokens, max_logit, lse, w, st);
  return head_impl<float>(h, hidden, rows, temperature, tokens, max_logit, lse, w, st);
}

dflash_status dflash_verify_greedy(dflash_handle h, const int32_t* draft,
                                   const void* target_logits, int32_t batch, int32_t* out_tokens,
                                   int32_t* n_accepted, int32_t* n_emitted, void* ws,
                                   size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (batch < 0) return fail(DFLASH_EINVAL, "batch < 0");
  if (batch == 0) return DFLASH_OK;
  NEED(draft, "draft");
  NEED(target_logits, "target_logits");
  NEED(out_tokens, "out_tokens");
  NEED(n_accepted, "n_accepted");
  NEED(n_emitted, "n_emitted");
  const int S = h->c.block_size, V = h->c.vocab, rows = batch * S;
  if (S > 64) return fail(DFLASH_EUNSUPPORTED, "block_size > 64");
  if (rows > 65535) return fail(DFLASH_EUNSUPPORTED, "batch*block_size > 65535");
  Carve cv{static_cast<char*>(ws)};
  VerifyWs w = carve_verify(h, cv, batch, false);
  TRY(check_ws(ws, ws_bytes, cv.off));
  const int nch = verify_chunks(h, rows), chunk = chunk_of(h, nch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->bf16)
    return launch(k_verify_greedy<bf16>, dim3(nch, rows), dim3(kRowThreads), 0, st,
                  static_cast<const bf16*>(target_logits), draft, S, V, chunk, w.pv, w.pi, w.ctl,
                  out_tokens, n_accepted, n_emitted, h->d_err, 0);
  return launch(k_verify_greedy<float>, dim3(nch, rows), dim3(kRowThreads), 0, st,
                static_cast<const float*>(target_logits), draft, S, V, chunk, w.pv, w.pi, w.ctl,
                out_tokens, n_accepted, n_emitted, h->d_err, 0);
}

dflash_status dflash_verify_sample(dflash_handle h, const int32_t* draft, const void* final_hidden,
                                   const float* draft_max, const float* draft_lse,
                                   const void* target_logits, const float* uniforms,
                                   float temperature, int32_t batch, int32_t* out_tokens,
                                   int32_t* n_accepted, int32_t* n_emitted, void* ws,
                                   size_t ws_bytes, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (batch < 0) return fail(DFLASH_EINVAL, "batch < 0");
  if (!(temperature > 0.f)) return fail(DFLASH_EINVAL, "temperature must be > 0");
  if (batch == 0) return DFLASH_OK;
  NEED(draft, "draft");
  NEED(final_hidden, "final_hidden");
  NEED(draft_max, "draft_max");
  NEED(draft_lse, "draft_lse");
  NEED(target_logits, "target_logits");
  NEED(uniforms, "uniforms");
  NEED(out_tokens, "out_tokens");
  NEED(n_accepted, "n_accepted");
  NEED(n_emitted, "n_emitted");
  const int rows = batch * h->c.block_size;
  if (rows > 65535 || rows + batch > 2 * kTileWords) return fail(DFLASH_EUNSUPPORTED, "batch too large");
  Carve cv{static_cast<char*>(ws)};
  VerifyWs w = carve_verify(h, cv, batch, true);
  TRY(check_ws(ws, ws_bytes, cv.off));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->bf16)
    return sample_impl<bf16>(h, draft, final_hidden, draft_max, draft_lse, target_logits, uniforms,
                             temperature, batch, out_tokens, n_accepted, n_emitted, w, st);
  return sample_impl<float>(h, draft, final_hidden, draft_max, draft_lse, target_logits, uniforms,
                            temperature, batch, out_tokens, n_accepted, n_emitted, w, st);
}

dflash_status dflash_get_device_error(dflash_handle h, int32_t* code, int32_t clear) {
  if (!code) return fail(DFLASH_EINVAL, "null argument");
  CHECK_HANDLE(h);
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemcpy(code, h->d_err, sizeof(int), cudaMemcpyDeviceToHost));
  if (clear) CUDA_TRY(cudaMemset(h->d_err, 0, sizeof(int)));
  return DFLASH_OK;
}

dflash_status dflash_fp8_packed_bytes(int32_t rows, int32_t cols, size_t* bytes) {
  if (!bytes || rows <= 0 || cols <= 0) return fail(DFLASH_EINVAL, "bad arguments");
  *bytes = fp8_packed_bytes(rows, cols);
  return DFLASH_OK;
}

dflash_status dflash_pack_fp8(const void* w, int32_t rows, int32_t cols, void* packed,
                              void* stream) {
  g_launches = 0;
  if (rows <= 0 || cols <= 0) return fail(DFLASH_EINVAL, "bad sizes");
  NEED(w, "w");
  NEED(packed, "packed");
  uint8_t* codes = static_cast<uint8_t*>(packed);
  float* scales = reinterpret_cast<float*>(codes + fp8_scale_offset(rows, cols));
  return launch(k_pack_fp8, dim3(rows), dim3(kRowThreads), 0, static_cast<cudaStream_t>(stream),
                static_cast<const bf16*>(w), cols, codes, static_cast<int>(fp8_ld(cols)), scales);
}

dflash_status dflash_test_force_timeout(dflash_handle h, int32_t enable) {
  CHECK_HANDLE(h);
  h->force_timeout = enable != 0;
  return DFLASH_OK;
}

}  // extern "C"

// ------------------------------------------------- greedy verification, no allocation
// Some callers cannot allocate device memory where they verify a block: a host runtime
// that hands out only buffers it already owns, code running under a frozen memory
// budget where cudaMalloc is forbidden, or a plain C caller with no allocator at all.
// dflash_verify_greedy_static serves them with the same kernel and the same results as
// dflash_verify_greedy; its scratch (per-chunk partial argmaxes and per-sequence
// counters) lives in one fixed device array of this library.
namespace {
constexpr size_t kStaticScratchBytes = 256 * 1024;  // per device, held until exit
constexpr int kStaticMaxRows = 16384;               // batch * block_size
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
std::mutex g_static_mu;
void* g_static_ptr[256] = {};  // device address of g_static_scratch, per device

// In host code the array's name only stands in for it; its device address is looked
// up once per device, with that device current, on the first call there.
dflash_status static_scratch(void** out) {
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 256) return fail(DFLASH_EUNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(DFLASH_ECUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return DFLASH_OK;
}
}  // namespace

extern "C" dflash_status dflash_verify_greedy_static(dflash_handle h, const int32_t* draft,
                                                     const void* target_logits, int32_t batch,
                                                     int32_t* out_tokens, int32_t* n_accepted,
                                                     int32_t* n_emitted, void* stream) {
  g_launches = 0;
  CHECK_HANDLE(h);
  if (batch < 0) return fail(DFLASH_EINVAL, "batch < 0");
  if (batch == 0) return DFLASH_OK;
  NEED(draft, "draft");
  NEED(target_logits, "target_logits");
  NEED(out_tokens, "out_tokens");
  NEED(n_accepted, "n_accepted");
  NEED(n_emitted, "n_emitted");
  const int S = h->c.block_size, V = h->c.vocab;
  if (S > 64) return fail(DFLASH_EUNSUPPORTED, "block_size > 64");
  if ((long long)batch * S > kStaticMaxRows)
    return fail(DFLASH_EUNSUPPORTED,
                "batch*block_size = %lld exceeds the static scratch limit of %d rows",
                (long long)batch * S, kStaticMaxRows);
  const int rows = batch * S;
  const int nch = verify_chunks(h, rows), chunk = chunk_of(h, nch);
  // layout: counters [batch], partial values [rows*nch], partial indices [rows*nch]
  const size_t off_v = ((size_t)batch * 4 + 255) & ~size_t(255);
  const size_t off_i = (off_v + (size_t)rows * nch * 4 + 255) & ~size_t(255);
  const size_t need = off_i + (size_t)rows * nch * 4;
  if (need > kStaticScratchBytes)
    return fail(DFLASH_EUNSUPPORTED, "static scratch too small: %zu > %zu bytes", need,
                kStaticScratchBytes);
  void* base = nullptr;
  TRY(static_scratch(&base));
  char* b = static_cast<char*>(base);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the counters must start at zero whatever an earlier call left in the array
  CUDA_TRY(cudaMemsetAsync(b, 0, (size_t)batch * 4, st));
  int* ctr = reinterpret_cast<int*>(b);
  float* pv = reinterpret_cast<float*>(b + off_v);
  int* pi = reinterpret_cast<int*>(b + off_i);
  if (h->bf16)
    return launch(k_verify_greedy<bf16>, dim3(nch, rows), dim3(kRowThreads), 0, st,
                  static_cast<const bf16*>(target_logits), draft, S, V, chunk, pv, pi, ctr,
                  out_tokens, n_accepted, n_emitted, h->d_err, 0);
  return launch(k_verify_greedy<float>, dim3(nch, rows), dim3(kRowThreads), 0, st,
                static_cast<const float*>(target_logits), draft, S, V, chunk, pv, pi, ctr,
                out_tokens, n_accepted, n_emitted, h->d_err, 0);
}
