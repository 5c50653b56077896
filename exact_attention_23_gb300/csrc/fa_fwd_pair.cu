// Instantiations and launch of the CTA-pair attention forward (head dim 64): clusters of two
// CTAs, launched as a programmatic dependent of the previous kernel on the stream.
#include <algorithm>
#include <atomic>

#include "fa_fwd_pair_kernel.cuh"
#include "fa_launch.h"

namespace fa {

// Clusters of two CTAs that can be resident at once (per device, found once): a cluster's
// CTAs must sit in one GPC, so GPCs with an odd number of free SMs leave one out, and a
// persistent grid larger than this would run a second wave.
static int max_pair_clusters(const void* fn, int smem) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int v = cached[dev].load(std::memory_order_acquire);
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached[dev].store(n, std::memory_order_release);
  return n;
}

template <bool CAUSAL>
static cudaError_t launch_pair(const FwdLaunch& a) {
  auto* fn = &fa_fwd_pair_kernel<CAUSAL>;
  const int smem = CfgP::kSmemBytes;
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
  const int clusters = max_pair_clusters(reinterpret_cast<const void*>(fn), smem);
  if (clusters <= 0) return cudaErrorLaunchFailure;
  const unsigned grid = std::min(a.grid, 2u * static_cast<unsigned>(clusters));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
}

cudaError_t launch_fwd_pair_d64(const FwdLaunch& a, bool causal) {
  return causal ? launch_pair<true>(a) : launch_pair<false>(a);
}

}  // namespace fa
