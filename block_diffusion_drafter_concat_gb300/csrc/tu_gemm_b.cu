// mma.sync GEMM kernel instantiations with 64 activation rows per tile, and the fp32
// SIMT kernels.
#include "host.h"

namespace dflash {

template <int BN>
static dflash_status by_epi(int epi, const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g,
                            int grid, const EpiArgs<bf16>& e, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch_tc<BN, EPI_F32>(tmA, wm, g, grid, e, st);
    case EPI_QKV: return launch_tc<BN, EPI_QKV>(tmA, wm, g, grid, e, st);
    case EPI_KV: return launch_tc<BN, EPI_KV>(tmA, wm, g, grid, e, st);
    case EPI_RESID: return launch_tc<BN, EPI_RESID>(tmA, wm, g, grid, e, st);
    case EPI_SWIGLU: return launch_tc<BN, EPI_SWIGLU>(tmA, wm, g, grid, e, st);
    case EPI_ARGMAX: return launch_tc<BN, EPI_ARGMAX>(tmA, wm, g, grid, e, st);
    case EPI_ARGKEY: return launch_tc<BN, EPI_ARGKEY>(tmA, wm, g, grid, e, st);
  }
  return fail(DFLASH_EUNSUPPORTED, "unknown epilogue %d", epi);
}

dflash_status launch_gemm_tc_hi(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st) {
  if (bn == 64) return by_epi<64>(epi, tmA, wm, g, grid, e, st);
  return fail(DFLASH_EUNSUPPORTED, "mma.sync tile with %d rows", bn);
}

dflash_status launch_gemm_f32(int epi, dim3 grid, const float* A, int lda, const WPtrs& w,
                              const GemmShape& g, const EpiArgs<float>& e, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch(k_gemm_f32<EPI_F32>, grid, dim3(256), 0, st, A, lda, w, g, e);
    case EPI_QKV: return launch(k_gemm_f32<EPI_QKV>, grid, dim3(256), 0, st, A, lda, w, g, e);
    case EPI_KV: return launch(k_gemm_f32<EPI_KV>, grid, dim3(256), 0, st, A, lda, w, g, e);
    case EPI_RESID: return launch(k_gemm_f32<EPI_RESID>, grid, dim3(256), 0, st, A, lda, w, g, e);
    case EPI_SWIGLU: return launch(k_gemm_f32<EPI_SWIGLU>, grid, dim3(256), 0, st, A, lda, w, g, e);
    case EPI_ARGMAX: return launch(k_gemm_f32<EPI_ARGMAX>, grid, dim3(256), 0, st, A, lda, w, g, e);
  }
  return fail(DFLASH_EUNSUPPORTED, "unknown epilogue %d", epi);
}

}  // namespace dflash
