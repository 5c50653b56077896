// Instantiations of the decode kernel (one query row per head, CUDA cores) and its launch,
// followed by the merge of key-range partial results when the keys are split.
#include "fa_launch.h"

namespace fa {

cudaError_t launch_decode(const DecodeParams& p, int d, unsigned combine_grid,
                          cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.n_splits);
  if (d == 64) fa_decode_kernel<64><<<grid, kDecThreads, 0, stream>>>(p);
  else fa_decode_kernel<128><<<grid, kDecThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  if (d == 64)
    fa_fwd_combine_kernel<64><<<combine_grid, 256, 0, stream>>>(p.o_part, p.lse_part, p.o, p.lse,
                                                                p.n_splits, p.BH);
  else
    fa_fwd_combine_kernel<128><<<combine_grid, 256, 0, stream>>>(p.o_part, p.lse_part, p.o, p.lse,
                                                                 p.n_splits, p.BH);
  return cudaGetLastError();
}

}  // namespace fa
