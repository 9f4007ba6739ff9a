// GEMM kernel instantiations with FP8 e4m3 weights (per-row scales) and 16 or 32
// activation rows per tile: the weight-streaming regime, where halving the weight bytes
// halves the time.
#include "host.h"

namespace dflash {

template <int BN>
static dflash_status by_epi(int epi, const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g,
                            int grid, const EpiArgs<bf16>& e, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch_tc<BN, EPI_F32, true>(tmA, wm, g, grid, e, st);
    case EPI_QKV: return launch_tc<BN, EPI_QKV, true>(tmA, wm, g, grid, e, st);
    case EPI_KV: return launch_tc<BN, EPI_KV, true>(tmA, wm, g, grid, e, st);
    case EPI_RESID: return launch_tc<BN, EPI_RESID, true>(tmA, wm, g, grid, e, st);
    case EPI_SWIGLU: return launch_tc<BN, EPI_SWIGLU, true>(tmA, wm, g, grid, e, st);
    case EPI_ARGMAX: return launch_tc<BN, EPI_ARGMAX, true>(tmA, wm, g, grid, e, st);
    case EPI_ARGKEY: return launch_tc<BN, EPI_ARGKEY, true>(tmA, wm, g, grid, e, st);
  }
  return fail(DFLASH_EUNSUPPORTED, "unknown epilogue %d", epi);
}

dflash_status launch_gemm_tc_f8(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st) {
  if (bn == 16) return by_epi<16>(epi, tmA, wm, g, grid, e, st);
  if (bn == 32) return by_epi<32>(epi, tmA, wm, g, grid, e, st);
  return fail(DFLASH_EUNSUPPORTED, "FP8 weights: tiles of 16 or 32 activation rows only");
}

}  // namespace dflash
