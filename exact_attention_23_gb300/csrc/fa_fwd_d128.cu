// Instantiations of the attention forward kernel for head dim 128.
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL>
static cudaError_t launch_one(const FwdLaunch& a) {
  auto* fn = &fa_fwd_kernel<D, CAUSAL>;
  const int smem = Cfg<D>::kSmemBytes;
  // Idempotent and cheap; done per call so that every device a caller uses is covered.
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fn<<<a.grid, kThreads, smem, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_d128(const FwdLaunch& a, bool causal) {
  return causal ? launch_one<128, true>(a) : launch_one<128, false>(a);
}

}  // namespace fa
