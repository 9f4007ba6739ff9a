// tcgen05 projection kernel instantiations on SM pairs (clusters of two CTAs, whole
// tiles): 128 and 256 activation rows per tile, every epilogue.
#include "host.h"
#include "umma.cuh"

namespace dflash {

template <int BN, int EPI>
static dflash_status launch_um2(const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g,
                                int grid, const EpiArgs<bf16>& e, cudaStream_t st) {
  using C = UmCfg<BN, true>;
  static std::atomic<unsigned long long> done{0};
  DFLASH_TRY(set_smem_once(k_gemm_umma<BN, EPI, true>, C::SMEM, done));
  return launch_pairs(k_gemm_umma<BN, EPI, true>, dim3(grid), dim3(C::THREADS), C::SMEM, st,
                      tmA, wm, g, e);
}

template <int BN>
static dflash_status by_epi2(int epi, const CUtensorMap& tmA, const WMaps& wm, const GemmShape& g,
                             int grid, const EpiArgs<bf16>& e, cudaStream_t st) {
  switch (epi) {
    case EPI_F32: return launch_um2<BN, EPI_F32>(tmA, wm, g, grid, e, st);
    case EPI_QKV: return launch_um2<BN, EPI_QKV>(tmA, wm, g, grid, e, st);
    case EPI_KV: return launch_um2<BN, EPI_KV>(tmA, wm, g, grid, e, st);
    case EPI_RESID: return launch_um2<BN, EPI_RESID>(tmA, wm, g, grid, e, st);
    case EPI_SWIGLU: return launch_um2<BN, EPI_SWIGLU>(tmA, wm, g, grid, e, st);
    case EPI_ARGMAX: return launch_um2<BN, EPI_ARGMAX>(tmA, wm, g, grid, e, st);
    case EPI_ARGKEY: return launch_um2<BN, EPI_ARGKEY>(tmA, wm, g, grid, e, st);
  }
  return fail(DFLASH_EUNSUPPORTED, "unknown epilogue %d", epi);
}

dflash_status launch_gemm_umma_pairs(int bn, int epi, const CUtensorMap& tmA, const WMaps& wm,
                                     const GemmShape& g, int grid, const EpiArgs<bf16>& e,
                                     cudaStream_t st) {
  if (bn == 128) return by_epi2<128>(epi, tmA, wm, g, grid, e, st);
  if (bn == 256) return by_epi2<256>(epi, tmA, wm, g, grid, e, st);
  return fail(DFLASH_EUNSUPPORTED, "tcgen05 pair tile with %d rows", bn);
}

}  // namespace dflash
