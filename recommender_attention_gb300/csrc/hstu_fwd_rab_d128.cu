// Instantiations of the persistent HSTU forward with a relative attention bias,
// head dimension 128.
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

static_assert(FwdCfg<128, 128, false, true>::SMEM_BYTES + sizeof(FwdSmemCtl) <= 232448, "shared memory over the per-CTA limit");
static_assert(FwdCfg<128, 128, true, true>::SMEM_BYTES + sizeof(FwdSmemCtl) <= 232448, "shared memory over the per-CTA limit");

namespace {
template <bool BF16, bool SOFTMAX>
cudaError_t launch_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q8,
                       const FwdParams& p, int grid, cudaStream_t stream) {
  constexpr int smem = FwdCfg<128, 128, SOFTMAX, true>::SMEM_BYTES;
  auto kern = hstu_fwd_kernel<128, 128, BF16, SOFTMAX, true>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_done[64] = {};
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  // programmatic dependent of the scheduler kernel launched just before it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, q8, p);
}
}  // namespace

cudaError_t launch_fwd_rab_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& q8, const FwdParams& p, bool bf16, bool softmax, int grid,
                               cudaStream_t stream) {
  if (bf16) return softmax ? launch_one<true, true>(q, k, v, q8, p, grid, stream)
                           : launch_one<true, false>(q, k, v, q8, p, grid, stream);
  return softmax ? launch_one<false, true>(q, k, v, q8, p, grid, stream)
                 : launch_one<false, false>(q, k, v, q8, p, grid, stream);
}

}  // namespace hstu
