// Instantiations of the HSTU backward with a relative attention bias, head dimension 64.
#include "hstu_bwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

static_assert(BwdCfg<64, 64, true>::SMEM_BYTES + sizeof(BwdCtl) <= 232448, "shared memory over the per-CTA limit");

cudaError_t launch_bwd_rab_d64(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q,
                               int grid_kv, cudaStream_t stream) {
  return launch_bwd_dispatch<64, 64, true>(m, p, bf16, softmax, grid_q, grid_kv, stream);
}

}  // namespace hstu
