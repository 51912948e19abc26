// Instantiations of the HSTU backward with a relative attention bias, head
// dimension 96 of q/k with hdim_v 96 or 64.
#include "hstu_bwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

static_assert(BwdCfg<96, 96, true>::SMEM_BYTES + sizeof(BwdCtl) <= 232448, "shared memory over the per-CTA limit");
static_assert(BwdCfg<96, 64, true>::SMEM_BYTES + sizeof(BwdCtl) <= 232448, "shared memory over the per-CTA limit");

cudaError_t launch_bwd_rab_d96(const BwdMaps& m, const BwdParams& p, int hdim_v, bool bf16, bool softmax, int grid_q,
                               int grid_kv, cudaStream_t stream) {
  return hdim_v == 64 ? launch_bwd_dispatch<96, 64, true>(m, p, bf16, softmax, grid_q, grid_kv, stream)
                      : launch_bwd_dispatch<96, 96, true>(m, p, bf16, softmax, grid_q, grid_kv, stream);
}

}  // namespace hstu
