// Internal interface between the host API (fa_api.cu) and the kernel instantiations
// (fa_fwd_d64.cu, fa_fwd_d128.cu, fa_bwd_d64.cu). Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_bwd_kernel.cuh"
#include "fa_decode_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_fwd1_kernel.cuh"
#include "fa_fwd_pair_kernel.cuh"

namespace fa {

constexpr int kMaxDevices = 64;

// Launches kernel<<<grid, block, smem, stream>>>(args...) as a programmatic dependent of
// the previous kernel on the stream: its launch and set-up overlap that kernel's tail, and
// the kernel waits for it with pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct FwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v;
  CUtensorMap tm_o;  // the output, boxes of 64 columns × 32 rows (one warp's rows)
  FwdParams p;
  unsigned grid;
  cudaStream_t stream;
};

// Each returns the CUDA error of the launch (cudaSuccess when enqueued).
cudaError_t launch_fwd_d64(const FwdLaunch& a, bool causal);
cudaError_t launch_fwd_d128(const FwdLaunch& a, bool causal);
// Q and K as e4m3 codes (tensor maps over bytes), d ∈ {64, 128}.
cudaError_t launch_fwd_fp8(const FwdLaunch& a, int d, bool causal);
// One 128-row Q tile per CTA with double-buffered S and P (fa_fwd1_kernel.cuh); a.p holds one
// tile per unit (tiles_per_cta = 1), d ∈ {64, 128}.
cudaError_t launch_fwd1(const FwdLaunch& a, int d, bool causal);
// The general form (queries against a longer key sequence, key ranges, block mask) on the
// one-tile kernel (tiles_per_cta = 1), then the merge when the key range is split.
cudaError_t launch_fwd1_gen(const FwdLaunch& a, int d, bool causal, unsigned combine_grid);
// Head dim 64 on CTA pairs (fa_fwd_pair_kernel.cuh): a.grid is even (clusters of two), a.p holds
// groups of four Q tiles per unit, tm_k has 64-row boxes and tm_v 32-column × 128-row boxes
// with the 64-byte swizzle.
cudaError_t launch_fwd_pair_d64(const FwdLaunch& a, bool causal);

// General form (Tq ≠ Tk, bottom-right causal, block masks, key ranges): the forward kernel
// with GEN = true, then, when a.p.n_splits > 1, the merge of the partial results.
cudaError_t launch_fwd_gen_d64(const FwdLaunch& a, bool causal, unsigned combine_grid);
cudaError_t launch_fwd_gen_d128(const FwdLaunch& a, bool causal, unsigned combine_grid);

// Decode (Tq = 1) on the CUDA cores: grid B·H × n_splits, then the merge when split.
cudaError_t launch_decode(const DecodeParams& p, int d, unsigned combine_grid,
                          cudaStream_t stream);
// Two query rows per head (Tq = kDecMultiMaxRows) on the CUDA cores, two warps per row: grid
// B·H × n_splits, then the merge when split. (From three rows on, the one-tile tensor-core
// kernel is faster.)
constexpr int kDecMultiMaxRows = 2;
cudaError_t launch_decode_multi(const DecodeParams& p, int d, unsigned combine_grid,
                                cudaStream_t stream);

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  BwdParams p;
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  float* lse2;
  float* dvec;
  __nv_bfloat16* dq;
  unsigned grid_main, grid_prep, grid_dq;
  cudaStream_t stream;
};

// Enqueues the three backward kernels (prep, main, dQ conversion) on a.stream.
cudaError_t launch_bwd_d64(const BwdLaunch& a, bool causal);
cudaError_t launch_bwd_d128(const BwdLaunch& a, bool causal);

}  // namespace fa
