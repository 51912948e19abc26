// Internal launchers shared by the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "hstu_common.cuh"

namespace hstu {

// Raises a kernel's dynamic shared-memory limit to `smem` bytes on the current
// device, once per device (devices 0..63; others set it on every call).
// `done` is one bit per device, owned by the caller's kernel instantiation.
// Safe from several host threads: two first calls may both set the attribute,
// which is harmless; a bit is published only after a successful set.
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel kern, int smem, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Tensor maps of the forward: q, k, v with 128-row boxes, q with 8-row boxes
// (query tiles whose rows come in two runs), o with 32-row boxes (the
// TMA-store epilogue) and k with 64-row boxes (the CTA-pair kernel, where each
// CTA loads half of a key tile); every box is 64 columns wide with a 128-byte
// swizzle.
struct FwdMaps {
  CUtensorMap q, k, v, q8, o, k64;
};
// Persistent forward over the scheduler's work units; one CTA per SM.
cudaError_t launch_fwd_d64(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                            cudaStream_t stream);
cudaError_t launch_fwd_d256(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                            cudaStream_t stream);
// hdim_qk 96 with hdim_v 96 or 64
cudaError_t launch_fwd_d96(const FwdMaps& m, const FwdParams& p, int hdim_v, bool bf16, bool softmax, int grid,
                           cudaStream_t stream);
// CTA pairs (hdim 128, no bias, in-kernel schedule: FwdParams::fused), on
// 2 x clusters CTAs; fwd_pair_max_clusters_d128 gives how many clusters fit on
// the device at once (0: none).
int fwd_pair_max_clusters_d128(bool bf16, bool softmax);
cudaError_t launch_fwd_pair_d128(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int clusters,
                                 cudaStream_t stream);
// with a relative attention bias (FwdParams::ts_q / rab_time / rab_pos)
cudaError_t launch_fwd_rab_d64(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                               cudaStream_t stream);
cudaError_t launch_fwd_rab_d96(const FwdMaps& m, const FwdParams& p, int hdim_v, bool bf16, bool softmax, int grid,
                               cudaStream_t stream);
cudaError_t launch_fwd_rab_d128(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                                cudaStream_t stream);
cudaError_t launch_fwd_rab_d256(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                                cudaStream_t stream);
// Tensor maps of the backward: 128-row boxes, and 8-row boxes for query tiles
// whose rows come in two runs.
struct BwdMaps {
  CUtensorMap q, k, v, d_o, q8, d_o8;
};
// dQ kernel then dK/dV kernel over the scheduler's query-tile and key-tile units.
cudaError_t launch_bwd_d64(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q, int grid_kv,
                           cudaStream_t stream);
cudaError_t launch_bwd_d128(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q, int grid_kv,
                            cudaStream_t stream);
// hdim_qk 96 with hdim_v 96 or 64
cudaError_t launch_bwd_d96(const BwdMaps& m, const BwdParams& p, int hdim_v, bool bf16, bool softmax, int grid_q,
                           int grid_kv, cudaStream_t stream);
// with a relative attention bias (BwdParams::ts_q / rab_time / rab_pos)
cudaError_t launch_bwd_rab_d64(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q,
                               int grid_kv, cudaStream_t stream);
cudaError_t launch_bwd_rab_d96(const BwdMaps& m, const BwdParams& p, int hdim_v, bool bf16, bool softmax, int grid_q,
                               int grid_kv, cudaStream_t stream);
cudaError_t launch_bwd_rab_d128(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q,
                                int grid_kv, cudaStream_t stream);
// delta[h, i] = sum_e dO[i, h, e] O[i, h, e] in fp32 over every row in [0, total_q).
cudaError_t launch_bwd_delta(const void* o, long long o_stride, const void* d_o, long long do_stride, float* delta,
                             int total_q, int nhead, int hdim_v, bool bf16, cudaStream_t stream);
cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);
// Zeroes the forward's workspace header (kWsHeaderInts ints) before a forward
// that schedules itself (FwdParams::fused).
cudaError_t launch_fwd_reset(int* ws_header, cudaStream_t stream);
// Split-KV merge (hdim_v 64, 96, 128 or 256), a programmatic dependent of the forward.
cudaError_t launch_combine(const CombineParams& p, int hdim, bool bf16, bool softmax, int sms, cudaStream_t stream);
cudaError_t launch_pairs(const PrepParams& p, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* result, unsigned long long timeout_ns, cudaStream_t stream);

}  // namespace hstu
