// Instantiations of the attention backward kernels for head dim 128.
#include <atomic>

#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL>
static cudaError_t launch_bwd(const BwdLaunch& a) {
  auto* fn = &fa_bwd_main_kernel<D, CAUSAL>;
  const int smem = BwdCfg<D>::kSmemBytes;
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
  // All three as programmatic dependents: each one's launch and set-up overlap the tail of
  // the kernel before it, and each waits for it (pdl_wait) before reading its results.
  cudaError_t e = launch_pdl(fa_bwd_prep_kernel<D>, a.grid_prep, 256, 0, a.stream, a.o, a.dout,
                             a.lse, a.lse2, a.dvec, a.p.dq_acc, a.p.T, a.p.T_pad, a.p.BH);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fn, a.grid_main, BwdCfg<D>::kThreads, smem, a.stream, a.tm_q, a.tm_k, a.tm_v, a.tm_do,
                 a.p);
  if (e != cudaSuccess) return e;
  return launch_pdl(fa_bwd_dq_kernel<D>, a.grid_dq, 256, 0, a.stream, a.p.dq_acc, a.dq, a.p.T,
                    a.p.n_qt, a.p.BH, a.p.scale);
}

cudaError_t launch_bwd_d128(const BwdLaunch& a, bool causal) {
  return causal ? launch_bwd<128, true>(a) : launch_bwd<128, false>(a);
}

}  // namespace fa
