// Instantiations of the decode kernel (one query row per head, CUDA cores) and its launch,
// followed by the merge of key-range partial results when the keys are split.
#include <atomic>

#include "fa_launch.h"

namespace fa {

namespace {

// The ring's shared-memory opt-in and a full shared-memory carveout (three 66 KB CTAs per
// SM) are per-device attributes: set once per device.
template <int D>
cudaError_t prepare_decode() {
  static std::atomic<uint64_t> done[kMaxDevices / 64 + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = 1ull << (dev % 64);
  if (done[dev / 64].load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fa_decode_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       dec_smem_bytes<D>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fa_decode_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           100);
  if (e != cudaSuccess) return e;
  done[dev / 64].fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int D, int KP>
cudaError_t prepare_decode_multi() {
  static std::atomic<uint64_t> done[kMaxDevices / 64 + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = 1ull << (dev % 64);
  if (done[dev / 64].load(std::memory_order_acquire) & bit) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fa_decode_multi_kernel<D, KP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       dec_smem_bytes<D>());
  if (e != cudaSuccess) return e;
  done[dev / 64].fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int D, int KP>
cudaError_t launch_multi(const DecodeParams& p, unsigned grid, cudaStream_t stream) {
  cudaError_t e = prepare_decode_multi<D, KP>();
  if (e != cudaSuccess) return e;
  return launch_pdl(fa_decode_multi_kernel<D, KP>, grid, kDecBlock, dec_smem_bytes<D>(), stream, p);
}


}  // namespace

cudaError_t launch_decode_multi(const DecodeParams& p, int d, unsigned combine_grid,
                                cudaStream_t stream) {
  constexpr int kKP = 2;  // warps per query row
  const int rows = kDecThreads / 32 / kKP;
  const int n_qblk = (p.Tq + rows - 1) / rows;
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.n_splits) *
                        static_cast<unsigned>(n_qblk);
  cudaError_t e = (d == 64) ? launch_multi<64, kKP>(p, grid, stream)
                            : launch_multi<128, kKP>(p, grid, stream);
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  const int out_rows = p.BH * p.Tq;
  const unsigned need = static_cast<unsigned>((static_cast<unsigned long long>(out_rows) + 7) / 8);
  const unsigned cg = need < combine_grid ? need : combine_grid;
  return (d == 64) ? launch_pdl(fa_fwd_combine_kernel<64>, cg, 256, 0, stream,
                                static_cast<const float*>(p.o_part), static_cast<const float*>(p.lse_part),
                                p.o, p.lse, p.n_splits, out_rows)
                   : launch_pdl(fa_fwd_combine_kernel<128>, cg, 256, 0, stream,
                                static_cast<const float*>(p.o_part), static_cast<const float*>(p.lse_part),
                                p.o, p.lse, p.n_splits, out_rows);
}

cudaError_t launch_decode(const DecodeParams& p, int d, unsigned combine_grid,
                          cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.n_splits);
  cudaError_t e = (d == 64) ? prepare_decode<64>() : prepare_decode<128>();
  if (e != cudaSuccess) return e;
  e = (d == 64) ? launch_pdl(fa_decode_kernel<64>, grid, kDecBlock, dec_smem_bytes<64>(), stream, p)
                : launch_pdl(fa_decode_kernel<128>, grid, kDecBlock, dec_smem_bytes<128>(), stream,
                             p);
  if (e != cudaSuccess || p.n_splits <= 1) return e;
  // one merge warp per row, 8 warps per block
  const unsigned need = static_cast<unsigned>((static_cast<unsigned long long>(p.BH) + 7) / 8);
  const unsigned cg = need < combine_grid ? need : combine_grid;
  const float* op = p.o_part;
  const float* lp = p.lse_part;
  return (d == 64) ? launch_pdl(fa_fwd_combine_kernel<64>, cg, 256, 0, stream, op, lp, p.o, p.lse,
                                p.n_splits, p.BH)
                   : launch_pdl(fa_fwd_combine_kernel<128>, cg, 256, 0, stream, op, lp, p.o, p.lse,
                                p.n_splits, p.BH);
}

}  // namespace fa
