// tcgen05 attention instantiation (head_dim 64).
#include "host.h"
#include "attn_umma.cuh"

namespace dflash {

template <int HD>
static dflash_status one(dim3 grid, const AuMaps& mp, const AttnArgs<bf16>& a, cudaStream_t st) {
  using C = AuCfg<HD>;
  static bool set = false;
  if (!set) {
    DFLASH_TRY(set_smem(k_attn_umma<HD>, C::SMEM));
    set = true;
  }
  return launch(k_attn_umma<HD>, grid, dim3(C::THREADS), C::SMEM, st, mp, a);
}

dflash_status launch_attn_umma(int hd, dim3 grid, const AuMaps& mp, const AttnArgs<bf16>& a,
                               cudaStream_t st) {
  if (hd == 64) return one<64>(grid, mp, a, st);
  return fail(DFLASH_EUNSUPPORTED, "tcgen05 attention: head_dim %d", hd);
}

}  // namespace dflash
