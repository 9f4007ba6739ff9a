// Host-side helpers shared by the translation units of libdflash: error reporting,
// kernel launches with programmatic dependent launch, and the per-unit launchers of
// the GEMM and attention kernels (each defined in its own translation unit so the
// kernel instantiations compile in parallel).
#pragma once

#include <cuda_runtime.h>

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

template <typename K>
dflash_status set_smem(K kern, int bytes) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return fail(DFLASH_ECUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  return DFLASH_OK;
}

template <int BN, int EPI>
dflash_status launch_tc(const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g, int grid,
                        const EpiArgs<bf16>& e, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    DFLASH_TRY(set_smem(k_gemm_tc<BN, EPI>, TcCfg<BN>::SMEM));
    attr_set = true;
  }
  return launch(k_gemm_tc<BN, EPI>, dim3(grid), dim3(TcCfg<BN>::THREADS), TcCfg<BN>::SMEM, st,
                tmA, wm, g, e);
}

// tu_gemm_a.cu: BN 16 and 32; tu_gemm_b.cu: BN 64 and the fp32 kernels;
// tu_attn.cu: attention.
dflash_status launch_gemm_tc_lo(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st);
dflash_status launch_gemm_tc_hi(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st);
// tu_gemm_c.cu: the tcgen05 kernel, 128 and 256 activation rows per tile
dflash_status launch_gemm_umma(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
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
