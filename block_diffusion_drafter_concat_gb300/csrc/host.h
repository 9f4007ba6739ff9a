// Host-side helpers shared by the translation units of libdflash: error reporting,
// kernel launches with programmatic dependent launch, and the per-unit launchers of
// the GEMM and attention kernels (each defined in its own translation unit so the
// kernel instantiations compile in parallel).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "attention.cuh"
#include "gemm.cuh"

namespace dflash {

dflash_status fail(dflash_status s, const char* fmt, ...);
void count_launch();

#define DFLASH_TRY(expr)                                                                 \
  do {                                                                                   \
    dflash_status s_ = (expr);                                                           \
    if (s_ != DFLASH_OK) return s_;                                                      \
  } while (0)

// Launches `kern` on `st`; the programmatic-stream-serialization attribute lets the
// kernel start while the previous kernel on the stream drains (see pdl_wait).
template <typename... KArgs, typename... Args>
dflash_status launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return fail(DFLASH_ECUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  count_launch();
  return DFLASH_OK;
}

// The same for clusters of two CTAs (SM pairs): the grid must be even.
template <typename... KArgs, typename... Args>
dflash_status launch_pairs(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t st, Args... args) {
  if (grid.x % 2 != 0) return fail(DFLASH_EINVAL, "SM-pair launch with an odd grid (%u)", grid.x);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return fail(DFLASH_ECUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  count_launch();
  return DFLASH_OK;
}

template <typename K>
dflash_status set_smem(K kern, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(DFLASH_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  return DFLASH_OK;
}

// cudaFuncSetAttribute applies to the current device only: `done` remembers, per kernel,
// the devices (bit = ordinal, below 64) it has been set on; higher ordinals set it on
// every launch.
template <typename K>
dflash_status set_smem_once(K kern, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DFLASH_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return DFLASH_OK;
  DFLASH_TRY(set_smem(kern, bytes));
  done.fetch_or(bit, std::memory_order_acq_rel);
  return DFLASH_OK;
}

template <int BN, int EPI, bool F8 = false>
dflash_status launch_tc(const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g, int grid,
                        const EpiArgs<bf16>& e, cudaStream_t st) {
  using C = TcCfg<BN, F8>;
  static std::atomic<unsigned long long> done{0};
  DFLASH_TRY(set_smem_once(k_gemm_tc<BN, EPI, F8>, C::SMEM, done));
  return launch(k_gemm_tc<BN, EPI, F8>, dim3(grid), dim3(C::THREADS), C::SMEM, st, tmA, wm, g,
                e);
}

// tu_gemm_a.cu: BN 16 and 32; tu_gemm_b.cu: BN 64 and the fp32 kernels;
// tu_attn.cu: attention.
dflash_status launch_gemm_tc_lo(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st);
dflash_status launch_gemm_tc_hi(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st);
// tu_gemm_f8.cu: FP8-weight instantiations, 16 and 32 activation rows per tile
dflash_status launch_gemm_tc_f8(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st);
// tu_gemm_c.cu: the tcgen05 kernel, 128 and 256 activation rows per tile
dflash_status launch_gemm_umma(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                               const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                               cudaStream_t st);
// tu_gemm_d.cu: the same on SM pairs (whole tiles, an even grid of CTAs)
dflash_status launch_gemm_umma_pairs(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                     const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                     cudaStream_t st);
dflash_status launch_gemm_f32(int epi, dim3 grid, const float* A, int lda, const WPtrs& w,
                              const GemmShape& g, const EpiArgs<float>& e, cudaStream_t st);
dflash_status launch_attn_tc(int hd, int nw, dim3 grid, int smem, const AttnMaps& mp,
                             const AttnArgs<bf16>& a, cudaStream_t st);
dflash_status launch_attn_f32(dim3 grid, int smem, const AttnArgs<float>& a, cudaStream_t st);
// tu_attn_umma.cu: tcgen05 attention (head_dim 64 with up to 128 query rows per kv head;
// key-split mode for up to 64 rows, head_dim 64 or 128)
dflash_status launch_attn_umma(int hd, bool ksplit, dim3 grid, const AuMaps& mp,
                               const AttnArgs<bf16>& a, cudaStream_t st);
dflash_status launch_attn_combine(int B, const AttnArgs<bf16>& a, cudaStream_t st);
dflash_status launch_attn_combine(int B, const AttnArgs<float>& a, cudaStream_t st);

}  // namespace dflash
