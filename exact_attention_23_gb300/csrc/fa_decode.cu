// Instantiations of the decode kernel (one query row per head, CUDA cores) and its launch,
// followed by the merge of key-range partial results when the keys are split.
#include "fa_launch.h"

namespace fa {

cudaError_t launch_decode(const DecodeParams& p, int d, unsigned combine_grid,
                          cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.n_splits);
  cudaError_t e = (d == 64) ? launch_pdl(fa_decode_kernel<64>, grid, kDecThreads, 0, stream, p)
                            : launch_pdl(fa_decode_kernel<128>, grid, kDecThreads, 0, stream, p);
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  // one merge thread per (row, 8 columns)
  const unsigned long long items = static_cast<unsigned long long>(p.BH) * (d / 8);
  const unsigned need = static_cast<unsigned>((items + 255) / 256);
  const unsigned cg = need < combine_grid ? need : combine_grid;
  const float* op = p.o_part;
  const float* lp = p.lse_part;
  return (d == 64) ? launch_pdl(fa_fwd_combine_kernel<64>, cg, 256, 0, stream, op, lp, p.o, p.lse,
                                p.n_splits, p.BH)
                   : launch_pdl(fa_fwd_combine_kernel<128>, cg, 256, 0, stream, op, lp, p.o, p.lse,
                                p.n_splits, p.BH);
}

}  // namespace fa
