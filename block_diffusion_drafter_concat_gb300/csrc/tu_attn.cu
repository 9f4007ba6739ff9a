// Attention kernel instantiations (head_dim 64 / 128, 1-8 query warps) and fp32 path.
#include "host.h"

namespace dflash {

template <int HD, int NW>
static dflash_status one(dim3 grid, int smem, const AttnMaps& mp, const AttnArgs<bf16>& a,
                         cudaStream_t st) {
  static std::atomic<unsigned long long> done{0};
  DFLASH_TRY(set_smem_once(k_attn_tc<HD, NW>, smem, done));
  return launch(k_attn_tc<HD, NW>, grid, dim3((NW + 1) * 32), smem, st, mp, a);
}

dflash_status launch_attn_tc(int hd, int nw, dim3 grid, int smem, const AttnMaps& mp,
                             const AttnArgs<bf16>& a, cudaStream_t st) {
  if (hd == 128) {
    switch (nw) {
      case 1: return one<128, 1>(grid, smem, mp, a, st);
      case 2: return one<128, 2>(grid, smem, mp, a, st);
      case 4: return one<128, 4>(grid, smem, mp, a, st);
      case 8: return one<128, 8>(grid, smem, mp, a, st);
    }
  } else if (hd == 64) {
    switch (nw) {
      case 1: return one<64, 1>(grid, smem, mp, a, st);
      case 2: return one<64, 2>(grid, smem, mp, a, st);
      case 4: return one<64, 4>(grid, smem, mp, a, st);
      case 8: return one<64, 8>(grid, smem, mp, a, st);
    }
  }
  return fail(DFLASH_EUNSUPPORTED, "attention: head_dim %d with %d query rows", hd, nw * 16);
}

dflash_status launch_attn_f32(dim3 grid, int smem, const AttnArgs<float>& a, cudaStream_t st) {
  static std::atomic<unsigned long long> done{0};
  DFLASH_TRY(set_smem_once(k_attn_f32, 160 * 1024, done));
  return launch(k_attn_f32, grid, dim3(128), smem, st, a);
}

template <typename T>
static dflash_status combine(int B, const AttnArgs<T>& a, cudaStream_t st) {
  dim3 grid((a.QR + 7) / 8, a.hkv, B);
  if (a.nsplit <= 4) return launch(k_attn_combine<T, 4>, grid, dim3(8 * a.hd / 4), 0, st, a);
  if (a.nsplit <= 8) return launch(k_attn_combine<T, 8>, grid, dim3(8 * a.hd / 4), 0, st, a);
  return launch(k_attn_combine<T, 16>, grid, dim3(8 * a.hd / 4), 0, st, a);
}
dflash_status launch_attn_combine(int B, const AttnArgs<bf16>& a, cudaStream_t st) {
  return combine(B, a, st);
}
dflash_status launch_attn_combine(int B, const AttnArgs<float>& a, cudaStream_t st) {
  return combine(B, a, st);
}

}  // namespace dflash
