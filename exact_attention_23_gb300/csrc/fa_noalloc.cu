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
#include <cuda.h>
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

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The driver's context queries, looked up once through the runtime (no link-time
// dependency on libcuda).
struct CtxFns {
  CtxGetCurrentFn current = nullptr;
  CtxGetIdFn id = nullptr;
};
const CtxFns& ctx_fns() {
  static std::once_flag once;
  static CtxFns f;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
            cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      f.current = reinterpret_cast<CtxGetCurrentFn>(a);
      f.id = reinterpret_cast<CtxGetIdFn>(b);
    }
    cudaGetLastError();
  });
  return f;
}

// The unique id of the calling thread's current context, or 0 if there is none yet.
unsigned long long current_ctx_id() {
  const CtxFns& f = ctx_fns();
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!f.current || !f.id || f.current(&c) != CUDA_SUCCESS || !c || f.id(c, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Per device: the reservation's address and the context it belongs to. A device reset
// destroys the context and with it the loaded module; the next call then sees another
// context id and looks the address up again.
struct Slot {
  void* ptr = nullptr;
  unsigned long long ctx = 0;
};
std::mutex g_mu;
Slot g_slot[fa::kMaxDevices];

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
    Slot& sl = g_slot[dev];
    const unsigned long long ctx = current_ctx_id();
    if (!sl.ptr || ctx == 0 || ctx != sl.ctx) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        sl = Slot{};
        return FA_ERR_LAUNCH;
      }
      sl.ptr = p;
      sl.ctx = current_ctx_id();  // the lookup made the device's context current
    }
    scratch = sl.ptr;
  }
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch,
                static_cast<size_t>(FA_BWD_NOALLOC_SCRATCH_BYTES), B, H, T, d, causal, scale,
                stream);
}
