// Instantiations of the persistent HSTU forward for head dimension 96 of q/k,
// with v/o of dimension 96 or 64 (the asymmetric 96/64 case).
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

cudaError_t launch_fwd_d96(const FwdMaps& m, const FwdParams& p, int hdim_v, bool bf16, bool softmax, int grid,
                           cudaStream_t stream) {
  if (hdim_v == 96) return launch_fwd_dispatch<96, 96, false>(m, p, bf16, softmax, grid, stream);
  if (hdim_v == 64) return launch_fwd_dispatch<96, 64, false>(m, p, bf16, softmax, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace hstu
