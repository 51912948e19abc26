// hstu_attn_fwd_static_ws: the forward with its scratch in a fixed device
// array of this library instead of a caller-provided workspace.  The call
// allocates nothing: the array below is placed by the module loader, its
// device address is looked up on a device's first call (and kept once the
// lookup has succeeded), and every later call only clears its header and hands
// it to hstu_attn_fwd.
#include <cuda_runtime.h>

#include <atomic>

#include "hstu_attn.h"
#include "hstu_common.cuh"

namespace {

static_assert(HSTU_STATIC_WS_BYTES % 256 == 0, "static scratch size");
static_assert(hstu::kWsHeaderInts * sizeof(int) <= HSTU_STATIC_WS_BYTES, "header fits");

// One scratch per device (each device's context holds its own copy of the
// module's __device__ variables).
static __device__ __align__(256) unsigned char g_static_ws[HSTU_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;

// Per device: the looked-up address, or nullptr while no lookup has succeeded.
std::atomic<void*> g_addr[kMaxDevices];

// Device address of g_static_ws on the current device.  Only a successful
// lookup is kept: a failed one (say, a first call made while the context could
// not answer) is retried on the next call.  Racing first calls may both look
// it up; they store the same address.  nullptr on failure.
void* static_ws_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* a = g_addr[dev].load(std::memory_order_acquire);
  if (a != nullptr) return a;
  if (cudaGetSymbolAddress(&a, g_static_ws) != cudaSuccess) {
    cudaGetLastError();   // reset the runtime's last error, so this failure shows up in no later check
    return nullptr;
  }
  g_addr[dev].store(a, std::memory_order_release);
  return a;
}

}  // namespace

extern "C" hstu_status hstu_attn_fwd_static_ws(const hstu_fwd_args* args, void* stream,
                                               const void** workspace_used) {
  if (!args) return HSTU_ERR_INVALID_ARG;
  size_t need = 0;
  const hstu_status st = hstu_attn_fwd_workspace_size(args, &need);
  if (st != HSTU_OK) return st;
  if (need > HSTU_STATIC_WS_BYTES) return HSTU_ERR_WORKSPACE;
  void* ws = static_ws_address();
  if (!ws) return HSTU_ERR_CUDA;
  // The work counter and the device error word must read zero until this
  // call's scheduler kernel has run; clear the whole header.
  if (cudaMemsetAsync(ws, 0, hstu::kWsHeaderInts * sizeof(int), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return HSTU_ERR_CUDA;
  hstu_fwd_args a = *args;
  a.workspace = ws;
  a.workspace_bytes = HSTU_STATIC_WS_BYTES;
  const hstu_status r = hstu_attn_fwd(&a, stream);
  if (r == HSTU_OK && workspace_used) *workspace_used = ws;
  return r;
}
