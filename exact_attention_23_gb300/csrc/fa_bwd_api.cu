// Host side of the C ABI's backward entry points (include/fa.h): workspace sizing,
// argument validation, tensor maps and the three launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "fa.h"
#include "fa_host.h"
#include "fa_launch.h"

using namespace fa::host;

extern "C" {

// Workspace: [BH][T_pad] fp32 −log2e·LSE, [BH][T_pad] fp32 D, [BH][T_pad][d] fp32 dQ accumulator,
// each section starting on a 256-byte boundary. Returns 0 for unsupported sizes.
size_t fa_bwd_workspace_size(int B, int H, int T, int d) {
  if (B <= 0 || H <= 0 || T <= 0 || (d != 64 && d != 128)) return 0;
  const long long BH = static_cast<long long>(B) * H;
  const long long T_pad = (static_cast<long long>(T) + 127) / 128 * 128;
  if (BH > INT32_MAX || T_pad > INT32_MAX || (T_pad / 128) * BH > INT32_MAX) return 0;
  auto up = [](unsigned long long x) { return (x + 255ull) / 256ull * 256ull; };
  const unsigned long long rows = static_cast<unsigned long long>(BH) * T_pad;
  if (rows > (1ull << 56) / (static_cast<unsigned long long>(d) + 2) / 4) return 0;
  return static_cast<size_t>(2 * up(rows * 4) + up(rows * d * 4));
}

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv, void* workspace,
              size_t workspace_bytes, int B, int H, int T, int d, int causal, float scale,
              int* status, unsigned long long timeout_ns, unsigned int flags, void* stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || T <= 0 || (d != 64 && d != 128)) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  if ((flags & ~static_cast<unsigned>(FA_FLAG_TEST_STARVE_Q)) != 0u) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_size(B, H, T, d);
  if (need == 0 || workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_kt = (static_cast<long long>(T) + 127) / 128;  // 128-key tiles
  const long long T_pad = n_kt * 128;
  const int bq = (d == 64) ? 128 : 64;                                // query tile rows
  const long long n_qt = T_pad / bq;
  const long long elems = BH * T * d;
  if (elems >= (1LL << 62) / 2) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * d * 2 >= (1LL << 40)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0u)
    return FA_ERR_MISALIGNED;
  // Outputs and workspace must not overlap any input or one another.
  const size_t tb = static_cast<size_t>(elems) * 2, lb = static_cast<size_t>(BH) * T * 4;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_bytes[6] = {tb, tb, tb, tb, tb, lb};
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {tb, tb, tb, need};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_INVALID_ARG;
  }

  int dev = -1, sms = 0;
  const int dst = check_device(&dev, &sms);
  if (dst != FA_OK) return dst;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_LAUNCH;

  fa::BwdLaunch a;
  if (!encode_map(enc, &a.tm_q, q, T, d, static_cast<int>(BH), bq) ||
      !encode_map(enc, &a.tm_k, k, T, d, static_cast<int>(BH)) ||
      !encode_map(enc, &a.tm_v, v, T, d, static_cast<int>(BH)) ||
      !encode_map(enc, &a.tm_do, dout, T, d, static_cast<int>(BH), bq))
    return FA_ERR_INVALID_ARG;
  auto up = [](size_t x) { return (x + 255u) / 256u * 256u; };
  const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(T_pad);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.lse2 = reinterpret_cast<float*>(ws);
  a.dvec = reinterpret_cast<float*>(ws + up(rows * 4));
  a.p.dq_acc = reinterpret_cast<float*>(ws + 2 * up(rows * 4));
  a.p.lse2 = a.lse2;
  a.p.dvec = a.dvec;
  a.p.dk = static_cast<__nv_bfloat16*>(dk);
  a.p.dv = static_cast<__nv_bfloat16*>(dv);
  a.p.status = status;
  a.p.T = T;
  a.p.T_pad = static_cast<int>(T_pad);
  a.p.BH = static_cast<int>(BH);
  a.p.n_qt = static_cast<int>(n_qt);
  a.p.n_kt = static_cast<int>(n_kt);
  // Heads per group: Q and dO (bf16) plus the fp32 dQ accumulator are 8·T·d bytes per
  // head; about 64 MB of them (half the 129 MB L2) per group.
  const long long per_head = 8LL * T_pad * d;
  a.p.head_group = static_cast<int>(std::max<long long>(1, std::min<long long>(BH, (64LL << 20) / per_head)));
  a.p.scale = scale;
  a.p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  a.p.timeout_ns = timeout_ns ? timeout_ns : 2000000000ull;
  a.p.flags = flags;
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dout = static_cast<const __nv_bfloat16*>(dout);
  a.lse = lse;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.grid_main = static_cast<unsigned>(n_kt * BH);
  // The two streaming kernels: a few resident blocks per SM, grid-stride loops.
  a.grid_prep = static_cast<unsigned>(sms) * 8u;
  a.grid_dq = static_cast<unsigned>(sms) * 8u;
  a.stream = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      (d == 64) ? fa::launch_bwd_d64(a, causal != 0) : fa::launch_bwd_d128(a, causal != 0);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, void* workspace,
           size_t workspace_bytes, int B, int H, int T, int d, int causal, float scale,
           void* stream) {
  return fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, T, d,
                   causal, scale, nullptr, 0ull, 0u, stream);
}

}  // extern "C"
