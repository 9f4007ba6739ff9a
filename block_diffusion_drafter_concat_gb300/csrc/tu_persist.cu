// The persistent layer-stack kernel: cooperative launch (all CTAs resident, required by
// its grid barriers) with programmatic stream serialization.
#define DFLASH_PERSIST_KERNEL
#include "host.h"

namespace dflash {

int persist_max_grid(int sms) {
  static int occ = -1;
  if (occ < 0) {
    if (cudaFuncSetAttribute(k_draft_persist, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_draft_persist, 160, kPSmem) !=
            cudaSuccess)
      occ = 0;
  }
  return occ > 0 ? sms : 0;
}

dflash_status launch_persist(int grid, const PersistMaps& maps, const PersistArgs& a,
                             cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(160);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_draft_persist, maps, a);
  if (e != cudaSuccess)
    return fail(DFLASH_ECUDA, "persistent kernel launch failed: %s", cudaGetErrorString(e));
  count_launch();
  return DFLASH_OK;
}

}  // namespace dflash
