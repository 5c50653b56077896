// Instantiations of the one-tile, double-buffered attention forward (head dims 64 and 128).
#include <atomic>

#include "fa_fwd1_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL>
static cudaError_t launch1(const FwdLaunch& a) {
  auto* fn = &fa_fwd1_kernel<D, CAUSAL>;
  const int smem = Cfg1<D>::kSmemBytes;
  // The shared-memory opt-in is a per-device attribute: set it once per device.
  static std::atomic<uint64_t> done[kMaxDevices / 64 + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = 1ull << (dev % 64);
  if (!(done[dev / 64].load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done[dev / 64].fetch_or(bit, std::memory_order_acq_rel);
  }
  return launch_pdl(fn, a.grid, Cfg1<D>::kThreads, smem, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
}

cudaError_t launch_fwd1(const FwdLaunch& a, int d, bool causal) {
  if (d == 64) return causal ? launch1<64, true>(a) : launch1<64, false>(a);
  return causal ? launch1<128, true>(a) : launch1<128, false>(a);
}

}  // namespace fa
