// GEMM kernel instantiations with 16 and 32 activation rows per tile.
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

dflash_status launch_gemm_tc_lo(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                cudaStream_t st) {
  if (bn == 16) return by_epi<16>(epi, tmA, wm, g, grid, e, st);
  return by_epi<32>(epi, tmA, wm, g, grid, e, st);
}

}  // namespace dflash
