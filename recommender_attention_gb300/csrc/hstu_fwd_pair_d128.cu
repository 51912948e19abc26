// Instantiations of the CTA-pair HSTU forward (head dimension 128).
#include "hstu_fwd_pair_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

int fwd_pair_max_clusters_d128(bool bf16, bool softmax) {
  if (bf16) return softmax ? fwd_pair_max_clusters<true, true>() : fwd_pair_max_clusters<true, false>();
  return softmax ? fwd_pair_max_clusters<false, true>() : fwd_pair_max_clusters<false, false>();
}

cudaError_t launch_fwd_pair_d128(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int clusters,
                                 cudaStream_t stream) {
  if (bf16) return softmax ? launch_fwd_pair_inst<true, true>(m, p, clusters, stream)
                           : launch_fwd_pair_inst<true, false>(m, p, clusters, stream);
  return softmax ? launch_fwd_pair_inst<false, true>(m, p, clusters, stream)
                 : launch_fwd_pair_inst<false, false>(m, p, clusters, stream);
}

}  // namespace hstu
