// Internal launchers shared by the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "hstu_common.cuh"

namespace hstu {

// Persistent forward over the scheduler's work units; one CTA per SM.  q8 is
// the q tensor map with 8-row boxes (query tiles whose rows come in two runs).
cudaError_t launch_fwd_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q8,
                           const FwdParams& p, bool bf16, bool softmax, int grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q8,
                            const FwdParams& p, bool bf16, bool softmax, int grid, cudaStream_t stream);
// hdim_qk 96 with hdim_v 96 or 64
cudaError_t launch_fwd_d96(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q8,
                           const FwdParams& p, int hdim_v, bool bf16, bool softmax, int grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q8,
                            const FwdParams& p, bool bf16, bool softmax, int grid, cudaStream_t stream);
cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);
cudaError_t launch_pairs(const PrepParams& p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int hdim, bool bf16, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* result, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace hstu
