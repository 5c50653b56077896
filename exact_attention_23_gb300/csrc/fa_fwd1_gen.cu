// Instantiations of the one-tile, double-buffered attention forward in its general form
// (head dims 64 and 128), and the merge of split key ranges.
#include <atomic>

#include "fa_fwd1_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL>
static cudaError_t launch1g(const FwdLaunch& a, unsigned combine_grid) {
  auto* fn = &fa_fwd1_kernel<D, CAUSAL, true>;
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
  cudaError_t e = launch_pdl(fn, a.grid, Cfg1<D>::kThreads, smem, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  if (e != cudaSuccess || a.p.n_splits <= 1) return e;
  const float* op = a.p.o_part;
  const float* lp = a.p.lse_part;
  return launch_pdl(fa_fwd_combine_kernel<D>, combine_grid, 256, 0, a.stream, op, lp, a.p.o,
                    a.p.lse, a.p.n_splits, a.p.BH * a.p.T);
}

cudaError_t launch_fwd1_gen(const FwdLaunch& a, int d, bool causal, unsigned combine_grid) {
  if (d == 64) return causal ? launch1g<64, true>(a, combine_grid) : launch1g<64, false>(a, combine_grid);
  return causal ? launch1g<128, true>(a, combine_grid) : launch1g<128, false>(a, combine_grid);
}

}  // namespace fa
