// Instantiations of the persistent HSTU forward for head dimension 64.
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

cudaError_t launch_fwd_d64(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                            cudaStream_t stream) {
  return launch_fwd_dispatch<64, 64, false>(m, p, bf16, softmax, grid, stream);
}

}  // namespace hstu
