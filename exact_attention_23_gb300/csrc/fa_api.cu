// Host side of the C ABI declared in include/fa.h, forward pass and shared helpers:
// argument validation, tensor-map encoding for the TMA loads, and the launch on the
// caller's stream. The backward's entry points are in fa_bwd_api.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <limits>
#include <mutex>

#include "fa.h"
#include "fa_host.h"
#include "fa_launch.h"

namespace fa {
namespace host {

// The driver's tensor-map encoder, looked up once through the runtime (no link-time
// dependency on libcuda).
EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

using fa::kMaxDevices;
// 0 = unknown, 1 = supported (cc 10.3), 2 = unsupported
static int g_dev_state[kMaxDevices];
static int g_dev_sms[kMaxDevices];
static std::mutex g_dev_mu;

int check_device(int* dev_out, int* sms_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return FA_ERR_UNSUPPORTED_DEVICE;
  }
  *dev_out = dev;
  if (dev >= kMaxDevices) return FA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_state[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_UNSUPPORTED_DEVICE;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_UNSUPPORTED_DEVICE;
    }
    g_dev_sms[dev] = sms;
    g_dev_state[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  *sms_out = g_dev_sms[dev];
  return g_dev_state[dev] == 1 ? FA_OK : FA_ERR_UNSUPPORTED_DEVICE;
}

// 3-D map over a [B·H][T][d] bf16 tensor: dim 0 = d (contiguous), dim 1 = T, dim 2 = B·H.
// Boxes are 64 columns (128 bytes, the 128-byte swizzle span) × box_rows rows × 1 head.
// Rows past T read as zeros, so a ragged last tile never touches the next head.
bool encode_map(EncodeTiledFn enc, CUtensorMap* map, const void* base, int T, int d, int BH,
                int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0u; }

float exponent_factor(double sl2, unsigned* negate) {
  *negate = sl2 < 0.0 ? fa::kIdescNegateA : 0u;
  if (sl2 == 0.0) return std::numeric_limits<float>::min();
  return static_cast<float>(sl2 < 0.0 ? -sl2 : sl2);
}

bool scale_ok(float scale) {
  return std::isfinite(scale) &&
         std::isfinite(static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074));
}

}  // namespace host
}  // namespace fa

using namespace fa::host;

namespace {

// 3-D map over [B·H][T][d] e4m3 codes (one byte each): one box of d bytes × 128 rows × 1
// head, swizzled in 128-byte (d = 128) or 64-byte (d = 64) rows.
bool encode_map_e4m3(EncodeTiledFn enc, CUtensorMap* map, const void* base, int T, int d,
                     int BH) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d),
                                 static_cast<cuuint64_t>(T) * static_cast<cuuint64_t>(d)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(d), 128, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
             elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
             d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over [B·H][T][64] bf16 values for the CTA-pair forward: boxes of 32 columns (64
// bytes, the 64-byte swizzle span) × 128 rows × 1 head; each CTA of a pair loads one half.
bool encode_map_v_half(EncodeTiledFn enc, CUtensorMap* map, const void* base, int T, int BH) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(T) * 128};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Validation, tensor maps and launch of the dense forward; qk8: q and k are e4m3 codes.
int dense_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                  int T, int d, int causal, float scale_log2, int* status,
                  unsigned long long timeout_ns, unsigned int flags, void* stream, bool qk8) {
  // ---- host-side validation: nothing is launched on failure
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || T <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale_log2)) return FA_ERR_INVALID_ARG;
  if ((flags & ~static_cast<unsigned>(FA_FLAG_TEST_STARVE_Q | FA_FLAG_TEST_STARVE_LATER_Q |
                                      FA_FLAG_CTA_PAIR)) != 0u)
    return FA_ERR_INVALID_ARG;
  const bool pair = (flags & FA_FLAG_CTA_PAIR) != 0u;
  if (pair && (d != 64 || qk8 || (flags & (FA_FLAG_TEST_STARVE_Q | FA_FLAG_TEST_STARVE_LATER_Q))))
    return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_qt = (static_cast<long long>(T) + 127) / 128;
  const long long n_pairs = (n_qt + 1) / 2;
  if (BH > INT32_MAX || n_qt * BH > INT32_MAX) return FA_ERR_INVALID_ARG;
  const long long elems = BH * T * d;
  if (elems >= (1LL << 62) / 2) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * d * 2 >= (1LL << 40)) return FA_ERR_INVALID_ARG;  // TMA stride limit
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  const size_t tbytes = static_cast<size_t>(elems) * 2;
  const size_t qkbytes = qk8 ? static_cast<size_t>(elems) : tbytes;
  const size_t lbytes = static_cast<size_t>(BH) * T * 4;
  if (overlaps(o, tbytes, q, qkbytes) || overlaps(o, tbytes, k, qkbytes) ||
      overlaps(o, tbytes, v, tbytes) || overlaps(lse, lbytes, q, qkbytes) ||
      overlaps(lse, lbytes, k, qkbytes) || overlaps(lse, lbytes, v, tbytes) ||
      overlaps(lse, lbytes, o, tbytes))
    return FA_ERR_INVALID_ARG;

  int dev = -1, sms = 0;
  const int dst = check_device(&dev, &sms);
  if (dst != FA_OK) return dst;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_LAUNCH;

  // Two 128-row Q tiles per CTA let the softmax of one overlap the MMAs of the other. When
  // pairs would leave SMs idle (short sequences), one tile per CTA runs instead; in bf16 that
  // is the kernel with double-buffered S and P (fa_fwd1_kernel.cuh), whose K steps overlap
  // within the tile (B4 H12 T512: 7.7 against 9.4 us, inputs in L2).
  const bool short_grid = n_pairs * BH < sms;
  const bool one = short_grid && !qk8 && !pair;
  const long long n_quads = (n_qt + 3) / 4;  // units of the CTA-pair kernel

  fa::FwdLaunch a;
  a.p = fa::FwdParams{};  // the general-form fields stay zero on this path
  const bool maps_ok =
      qk8 ? (encode_map_e4m3(enc, &a.tm_q, q, T, d, static_cast<int>(BH)) &&
             encode_map_e4m3(enc, &a.tm_k, k, T, d, static_cast<int>(BH)))
          : (encode_map(enc, &a.tm_q, q, T, d, static_cast<int>(BH)) &&
             encode_map(enc, &a.tm_k, k, T, d, static_cast<int>(BH)));
  if (pair && !(encode_map(enc, &a.tm_k, k, T, d, static_cast<int>(BH), 64) &&
                encode_map_v_half(enc, &a.tm_v, v, T, static_cast<int>(BH))))
    return FA_ERR_INVALID_ARG;
  if (!maps_ok || (!pair && !encode_map(enc, &a.tm_v, v, T, d, static_cast<int>(BH))) ||
      !encode_map(enc, &a.tm_o, o, T, d, static_cast<int>(BH), 32))
    return FA_ERR_INVALID_ARG;
  a.p.o = static_cast<__nv_bfloat16*>(o);
  a.p.lse = lse;
  a.p.status = status;
  a.p.T = T;
  a.p.BH = static_cast<int>(BH);
  const int tiles = (one || n_pairs * BH * 2 < sms) ? 1 : 2;
  const long long n_units = pair ? n_quads : (tiles == 2) ? n_pairs : n_qt;
  a.p.n_units = static_cast<int>(n_units);
  a.p.total_units = static_cast<int>(n_units * BH);
  // All heads interleaved in one cost-sorted list. (Limiting the interleave to the heads
  // whose K/V fit in L2 cut DRAM reads 2.6x at T = 16384 but measured 7-8 % slower: the
  // re-reads cost no time at < 20 % of HBM bandwidth, the coarser balance did.)
  a.p.div_bh = fa::FastDiv::make(static_cast<uint32_t>(BH));
  a.p.div_splits = fa::FastDiv::make(1u);
  a.p.tiles_per_cta = tiles;
  a.p.n_kv = static_cast<int>(n_qt);
  a.p.scale_log2 = exponent_factor(scale_log2, &a.p.s_negate);
  a.p.timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
  a.p.flags = flags;
  // Persistent: one CTA per SM (at most one per unit); each walks units blockIdx.x,
  // blockIdx.x + gridDim.x, ...
  a.grid = pair ? static_cast<unsigned>(2 * std::min<long long>(n_units * BH, sms / 2))
              : static_cast<unsigned>(std::min<long long>(n_units * BH, sms));
  a.stream = static_cast<cudaStream_t>(stream);

  const cudaError_t e = qk8   ? fa::launch_fwd_fp8(a, d, causal != 0)
                        : one ? fa::launch_fwd1(a, d, causal != 0)
                        : pair ? fa::launch_fwd_pair_d64(a, causal != 0)
                        : (d == 64) ? fa::launch_fwd_d64(a, causal != 0)
                                    : fa::launch_fwd_d128(a, causal != 0);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

const char* fa_version(void) { return "fa-gb300 0.1.0 sm_103a"; }

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_UNSUPPORTED_DEVICE: return "no CUDA device of compute capability 10.3 (sm_103a)";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_TIMEOUT: return "an internal wait of the kernel timed out";
    default: return "unknown status";
  }
}

int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int T, int d, int causal, float scale, int* status, unsigned long long timeout_ns,
              unsigned int flags, void* stream) {
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  return dense_forward(q, k, v, o, lse, B, H, T, d, causal,
                       static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074),
                       status, timeout_ns, flags, stream, false);
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* v, void* o, float* lse, float q_scale,
               float k_scale, int B, int H, int T, int d, int causal, float scale, void* stream) {
  for (float x : {q_scale, k_scale})
    if (!std::isfinite(x) || !(x > 0.0f)) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  const double sl2 = static_cast<double>(scale) * q_scale * k_scale * 1.4426950408889634074;
  return dense_forward(q8, k8, v, o, lse, B, H, T, d, causal, static_cast<float>(sl2), nullptr,
                       0ull, 0u, stream, true);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T,
           int d, int causal, float scale, void* stream) {
  return fa_fwd_ex(q, k, v, o, lse, B, H, T, d, causal, scale, nullptr, 0ull, 0u, stream);
}

}  // extern "C"
