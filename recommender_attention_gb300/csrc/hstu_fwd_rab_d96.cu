// Instantiations of the persistent HSTU forward with a relative attention bias,
// head dimension 96 of q/k with v/o of dimension 96 or 64.
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

cudaError_t launch_fwd_rab_d96(const FwdMaps& m, const FwdParams& p, int hdim_v, bool bf16, bool softmax, int grid,
                               cudaStream_t stream) {
  if (hdim_v == 96) return launch_fwd_dispatch<96, 96, true>(m, p, bf16, softmax, grid, stream);
  if (hdim_v == 64) return launch_fwd_dispatch<96, 64, true>(m, p, bf16, softmax, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace hstu
