// tcgen05 attention instantiations: head_dim 64 with 128 query rows per kv head, and
// head_dim 64 or 128 with at most 64 (key-split mode).
#include "host.h"
#include "attn_umma.cuh"

namespace dflash {

template <int HD, bool KSPLIT>
static dflash_status one(dim3 grid, const AuMaps& mp, const AttnArgs<bf16>& a, cudaStream_t st) {
  using C = AuCfg<HD, KSPLIT>;
  static std::atomic<unsigned long long> done{0};
  DFLASH_TRY(set_smem_once(k_attn_umma<HD, KSPLIT>, C::SMEM, done));
  return launch(k_attn_umma<HD, KSPLIT>, grid, dim3(C::THREADS), C::SMEM, st, mp, a);
}

dflash_status launch_attn_umma(int hd, bool ksplit, dim3 grid, const AuMaps& mp,
                               const AttnArgs<bf16>& a, cudaStream_t st) {
  if (hd == 64 && !ksplit) return one<64, false>(grid, mp, a, st);
  if (hd == 64 && ksplit) return one<64, true>(grid, mp, a, st);
  if (hd == 128 && ksplit) return one<128, true>(grid, mp, a, st);
  return fail(DFLASH_EUNSUPPORTED, "tcgen05 attention: head_dim %d", hd);
}

}  // namespace dflash
