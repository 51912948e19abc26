// Instantiations of the persistent HSTU forward with a relative attention bias,
// head dimension 256.
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

cudaError_t launch_fwd_rab_d256(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                                cudaStream_t stream) {
  return launch_fwd_dispatch<256, 256, true>(m, p, bf16, softmax, grid, stream);
}

}  // namespace hstu
