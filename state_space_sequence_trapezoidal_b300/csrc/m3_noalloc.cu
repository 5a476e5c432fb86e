// Prefill for callers that cannot allocate device memory.
//
// m3_ssm_prefill needs a small caller-owned workspace.  Some callers have no way
// to provide one: a plugin host or serving loop that forbids device allocation
// once it is running (cudaMalloc synchronises the device and can fail under
// memory pressure), or code that hands every byte of its budget to a pool it
// does not control.  m3_ssm_prefill_noalloc serves them from a scratch array that
// lives in this library's own device image: it is reserved when the library's
// module is loaded on a GPU and stays there until the process exits.
//
// The array's name in host code is only a host-side stand-in for the symbol, not
// a device address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "m3_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr on a CUDA error.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" m3_status m3_ssm_prefill_noalloc(const m3_dims* dims, const void* x, const void* B,
                                            const void* C, const void* dt, const float* A,
                                            const void* lambda, const void* theta,
                                            const m3_state* h0, void* y, const m3_state* hT,
                                            void* stream) {
  if (!dims) return M3_ERR_ARG;
  const size_t need = m3_ssm_prefill_workspace(dims);
  if (need > kStaticScratchBytes) return M3_ERR_WORKSPACE;
  void* ws = scratch_address();
  if (!ws) return M3_ERR_CUDA;
  // The workspace contract wants zeroed scratch on entry; the previous call (possibly one
  // whose bounded wait ran out) may have left a status bit behind.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return M3_ERR_CUDA;
  return m3_ssm_prefill(dims, x, B, C, dt, A, lambda, theta, h0, y, hT, ws, need, stream);
}
