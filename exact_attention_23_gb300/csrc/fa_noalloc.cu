// fa_bwd_noalloc: the backward pass with its workspace taken from a fixed reservation
// inside the library instead of from the caller.
//
// Some callers cannot hand the library a device buffer: a host program that has already
// given nearly all of the GPU's memory to its own pools, or one calling from a path where
// a device allocation is not acceptable (it can synchronise the device, and it can fail
// at run time, after the program has committed to the call). For them the workspace is a
// file-scope device array, reserved once when the library's device code is loaded. The
// array is reached through its symbol address; no allocation of any kind (cudaMalloc,
// cudaFree or an allocating library) happens here.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

// Nothing in it needs to start at zero: each call's first kernel writes the row
// statistics and zero-fills the dQ accumulator it uses.
static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[fa::kMaxDevices];  // per device; filled by the first call on it

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int T, int d, int causal, float scale,
                              void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_size(B, H, T, d);
  if (need == 0 || need > static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES))
    return FA_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fa::kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_UNSUPPORTED_DEVICE;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch,
                static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES), B, H, T, d, causal, scale,
                stream);
}
