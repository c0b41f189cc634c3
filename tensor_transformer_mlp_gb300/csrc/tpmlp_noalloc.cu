// tpmlp_backward_noalloc: the tensor-parallel MLP backward for callers that cannot allocate.
//
// tpmlp_backward keeps its n x m intermediate D = (G B^T) * gelu'(Z) in a workspace the
// caller allocates. Some callers cannot do that: a host that hands this library only the
// tensors of one step and owns no allocator on the device, code that must not allocate once
// its steady state has begun (allocation can block on a device-wide synchronisation or fail
// under fragmentation at an unpredictable moment), or a plugin whose host reserved all
// device memory up front. For them this file keeps D in a fixed scratch array in static
// device memory and runs the same backward on it. Nothing here calls cudaMalloc, cudaFree
// or any allocating routine.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tpmlp.h"
#include "tpmlp_internal.h"

namespace {

// Largest D this entry point can hold: 64 MiB (n * m * element size <= 67,108,864 bytes,
// e.g. n = 8192 tokens with m = 4096 in bf16). Every GPU that loads this code keeps the
// array for the life of the process.
constexpr size_t kScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_backward_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device
// (the host-side name of a __device__ array is only a stand-in for it). The address is cached
// by device number for the life of the process, so the array must stay where the first lookup
// found it: a cudaDeviceReset, or a context other than the device's primary one, is not
// supported (the library's per-device status word is cached the same way).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_backward_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" tpmlp_status tpmlp_backward_noalloc(const void* X, const void* A, const void* B, const void* G,
                                               const void* Z_save, const void* Y_save, void* dX, float* dA,
                                               float* dB, int64_t n, int64_t d, int64_t m, int t,
                                               tpmlp_gelu gelu, tpmlp_dtype dt, void* stream) {
  // The same argument checks as tpmlp_backward first, so that both entry points report the same
  // status for the same bad arguments; only then the size of D against the scratch array.
  const int st = tpmlp::validate_backward_args(X, A, B, G, Z_save, Y_save, dX, dA, dB, n, d, m, t, gelu, dt);
  if (st != TPMLP_OK) return static_cast<tpmlp_status>(st);
  const size_t need = tpmlp_backward_workspace_size(n, m, dt);
  if (need > kScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "tpmlp_backward_noalloc: D needs %zu bytes (n=%lld, m=%lld) but the static scratch holds %zu; "
             "use tpmlp_backward with a caller workspace",
             need, (long long)n, (long long)m, kScratchBytes);
    return static_cast<tpmlp_status>(tpmlp::report_error(TPMLP_ERR_WORKSPACE, msg));
  }
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[200];
      snprintf(msg, sizeof(msg), "tpmlp_backward_noalloc: scratch address lookup failed: %s", cudaGetErrorString(e));
      return static_cast<tpmlp_status>(tpmlp::report_error(TPMLP_ERR_CUDA, msg));
    }
  }
  // D is written in full by the first backward GEMM before anything reads it, so the scratch
  // needs no clearing between calls.
  return tpmlp_backward(X, A, B, G, Z_save, Y_save, dX, dA, dB, n, d, m, t, gelu, dt, scratch,
                        scratch ? kScratchBytes : 0, stream);
}
