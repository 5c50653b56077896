// Host side of the general-form forward entry points (include/fa.h): queries against a
// longer key sequence with the key range split over CTAs (fa_fwd_kv), and block-sparse
// self-attention (fa_fwd_block_sparse). Both run the forward kernel's general form.
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

namespace {

size_t round_up256(size_t x) { return (x + 255u) / 256u * 256u; }

// Key ranges per query tile when the caller asks for automatic choice. The units (query
// tile, range) run one per SM at a time, so a choice of s ranges costs about ⌈units·s / SMs⌉
// rounds of (K tiles per range + about one tile's worth of set-up and output). More ranges
// must be at least 5 % cheaper than fewer (partial rows and their merge cost memory
// traffic); at most 64.
int auto_splits(long long BH, long long n_qt, long long n_kt, int sms) {
  const long long units = BH * n_qt;
  long long best = 1, best_cost = -1;
  for (long long s = 1; s <= std::min<long long>(64, n_kt); ++s) {
    const long long per = (n_kt + s - 1) / s;
    const long long used = (n_kt + per - 1) / per;  // no empty range
    const long long cost = (units * used + sms - 1) / sms * (per + 1);
    if (best_cost < 0 || cost * 20 < best_cost * 19) {
      best_cost = cost;
      best = used;
    }
  }
  return static_cast<int>(best);
}

// Decode (one query row per head): as many key ranges as fit one wave of resident CTAs
// (a second, partial wave would double the time), each range at least 256 keys.
int decode_splits(long long BH, long long Tk, int sms) {
  long long s = static_cast<long long>(sms) * fa::kDecCtasPerSm / BH;
  s = std::min<long long>(s, std::max<long long>(1, Tk / 256));
  return static_cast<int>(std::max<long long>(1, std::min<long long>(s, 1024)));
}

// Two query rows (multi-query decode): two warps per row, two rows per CTA; key ranges so
// that B·H × ranges CTAs fill one wave (two per SM), each range at least 256 keys.
int multi_splits(long long BH, long long Tk, int sms) {
  long long s = static_cast<long long>(sms) * fa::kDecMultiCtasPerSm / BH;
  s = std::min<long long>(s, std::max<long long>(1, Tk / 256));
  return static_cast<int>(std::max<long long>(1, std::min<long long>(s, 1024)));
}

// Key ranges actually used for these sizes (requested > 0, or the automatic choice), with
// no empty range.
int effective_splits(long long BH, long long Tq, long long Tk, int requested, int sms) {
  const long long n_qt = (Tq + 127) / 128, n_kt = (Tk + 127) / 128;
  if (Tq <= fa::kDecMultiMaxRows) {
    long long s = requested ? requested
                            : (Tq == 1 ? decode_splits(BH, Tk, sms) : multi_splits(BH, Tk, sms));
    s = std::min<long long>(s, Tk);
    const long long per = (Tk + s - 1) / s;
    return static_cast<int>((Tk + per - 1) / per);
  }
  long long s = requested ? requested : auto_splits(BH, n_qt, n_kt, sms);
  s = std::min<long long>(s, n_kt);
  const long long per = (n_kt + s - 1) / s;
  return static_cast<int>((n_kt + per - 1) / per);
}

size_t partial_bytes(long long BH, long long Tq, int d, int splits) {
  if (splits <= 1) return 0;
  return round_up256(static_cast<size_t>(splits) * BH * Tq * d * 4) +
         round_up256(static_cast<size_t>(splits) * BH * Tq * 4);
}

struct GenArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  const uint8_t* bmask;
  int mask_heads;
  int B, H, Tq, Tk, d, causal;
  float scale;
  int splits;  // ≥ 1
  void* workspace;
  size_t workspace_bytes;
  void* stream;
  int* status;
  unsigned long long timeout_ns;
};

int launch_general(const GenArgs& g, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return FA_ERR_LAUNCH;
  const long long BH = static_cast<long long>(g.B) * g.H;
  const long long n_qt = (static_cast<long long>(g.Tq) + 127) / 128;
  const long long n_kt = (static_cast<long long>(g.Tk) + 127) / 128;
  fa::FwdLaunch a;
  a.p = fa::FwdParams{};
  if (!encode_map(enc, &a.tm_q, g.q, g.Tq, g.d, static_cast<int>(BH)) ||
      !encode_map(enc, &a.tm_k, g.k, g.Tk, g.d, static_cast<int>(BH)) ||
      !encode_map(enc, &a.tm_v, g.v, g.Tk, g.d, static_cast<int>(BH)) ||
      !encode_map(enc, &a.tm_o, g.o, g.Tq, g.d, static_cast<int>(BH), 32))
    return FA_ERR_INVALID_ARG;
  // Key ranges of equal length in K tiles; no range is empty.
  const long long per = (n_kt + g.splits - 1) / g.splits;
  const int splits = static_cast<int>((n_kt + per - 1) / per);
  // Two Q tiles per unit only when pairs still give every SM work.
  const long long n_pairs = (n_qt + 1) / 2;
  const int tiles = (n_qt >= 2 && n_pairs * BH * splits >= sms) ? 2 : 1;
  const long long n_units = (n_qt + tiles - 1) / tiles;
  if (n_units * splits * BH > INT32_MAX) return FA_ERR_INVALID_ARG;
  a.p.o = static_cast<__nv_bfloat16*>(g.o);
  a.p.lse = g.lse;
  a.p.status = g.status;
  a.p.T = g.Tq;
  a.p.BH = static_cast<int>(BH);
  a.p.n_units = static_cast<int>(n_units);
  a.p.total_units = static_cast<int>(n_units * splits * BH);
  a.p.n_kv = static_cast<int>(n_kt);
  a.p.tiles_per_cta = tiles;
  a.p.div_bh = fa::FastDiv::make(static_cast<uint32_t>(BH));
  a.p.scale_log2 = exponent_factor(static_cast<double>(g.scale) * 1.4426950408889634074,
                                   &a.p.s_negate);
  a.p.timeout_ns = g.timeout_ns ? g.timeout_ns : 2000000000ull;
  a.p.flags = 0u;
  a.p.Tk = g.Tk;
  a.p.n_qt = static_cast<int>(n_qt);
  a.p.kv_off = g.Tk - g.Tq;
  a.p.n_splits = splits;
  a.p.div_splits = fa::FastDiv::make(static_cast<uint32_t>(splits));
  a.p.kt_per_split = static_cast<int>(per);
  a.p.bmask = g.bmask;
  a.p.bmask_heads = g.mask_heads;
  a.p.o_part = nullptr;
  a.p.lse_part = nullptr;
  if (splits > 1) {
    uint8_t* ws = static_cast<uint8_t*>(g.workspace);
    a.p.o_part = reinterpret_cast<float*>(ws);
    a.p.lse_part = reinterpret_cast<float*>(
        ws + round_up256(static_cast<size_t>(splits) * BH * g.Tq * g.d * 4));
  }
  a.grid = static_cast<unsigned>(std::min<long long>(a.p.total_units, sms));
  a.stream = static_cast<cudaStream_t>(g.stream);
  const unsigned combine_grid = static_cast<unsigned>(sms) * 8u;
  // One Q tile per unit: the one-tile kernel, whose S and P are double-buffered, overlaps
  // consecutive K steps of its single tile.
  const cudaError_t e = (tiles == 1) ? fa::launch_fwd1_gen(a, g.d, g.causal != 0, combine_grid)
                        : (g.d == 64) ? fa::launch_fwd_gen_d64(a, g.causal != 0, combine_grid)
                                      : fa::launch_fwd_gen_d128(a, g.causal != 0, combine_grid);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Checks shared by both entry points; FA_OK when the arguments may be launched.
int validate_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    int B, int H, int Tq, int Tk, int d, float scale) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Tq <= 0 || Tk <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT32_MAX) return FA_ERR_INVALID_ARG;
  const long long Tmax = std::max(Tq, Tk);
  if (BH * Tmax * d >= (1LL << 62) / 2) return FA_ERR_INVALID_ARG;
  if (Tmax * d * 2 >= (1LL << 40)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  const size_t qb = static_cast<size_t>(BH) * Tq * d * 2, kb = static_cast<size_t>(BH) * Tk * d * 2;
  const size_t lb = static_cast<size_t>(BH) * Tq * 4;
  if (overlaps(o, qb, q, qb) || overlaps(o, qb, k, kb) || overlaps(o, qb, v, kb) ||
      overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
      overlaps(lse, lb, o, qb))
    return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_fwd_kv_workspace_size(int B, int H, int Tq, int Tk, int d, int n_splits) {
  if (B <= 0 || H <= 0 || Tq <= 0 || Tk <= 0 || (d != 64 && d != 128) || n_splits < 0)
    return 0;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_qt = (static_cast<long long>(Tq) + 127) / 128;
  const long long n_kt = (static_cast<long long>(Tk) + 127) / 128;
  (void)n_qt;
  (void)n_kt;
  int sms = 0;
  if (n_splits == 0) {
    int dev = -1;
    if (check_device(&dev, &sms) != FA_OK) return 0;
  }
  const int splits = effective_splits(BH, Tq, Tk, n_splits, sms);
  const size_t bytes = partial_bytes(BH, Tq, d, splits);
  return bytes == 0 ? 1 : bytes;  // nonzero: "supported, needs (almost) nothing"
}

int fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Tq, int Tk, int d, int causal, float scale, int n_splits, void* workspace,
              size_t workspace_bytes, void* stream) {
  int st = validate_common(q, k, v, o, lse, B, H, Tq, Tk, d, scale);
  if (st != FA_OK) return st;
  if (causal && Tq > Tk) return FA_ERR_INVALID_ARG;
  if (n_splits < 0) return FA_ERR_INVALID_ARG;
  int dev = -1, sms = 0;
  st = check_device(&dev, &sms);
  if (st != FA_OK) return st;
  const long long BH = static_cast<long long>(B) * H;
  const int splits = effective_splits(BH, Tq, Tk, n_splits, sms);
  const size_t need = partial_bytes(BH, Tq, d, splits);
  if (need > 0) {
    if (!workspace || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0u) return FA_ERR_MISALIGNED;
    const size_t qb = static_cast<size_t>(BH) * Tq * d * 2, kb = static_cast<size_t>(BH) * Tk * d * 2;
    if (overlaps(workspace, need, q, qb) || overlaps(workspace, need, k, kb) ||
        overlaps(workspace, need, v, kb) || overlaps(workspace, need, o, qb) ||
        overlaps(workspace, need, lse, static_cast<size_t>(BH) * Tq * 4))
      return FA_ERR_INVALID_ARG;
  }
  if (Tq == 1) {
    // One query row per head: a streaming kernel on the CUDA cores (the query sees every
    // key under bottom-right causal alignment, so causal changes nothing here).
    fa::DecodeParams dp{};
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.k = static_cast<const __nv_bfloat16*>(k);
    dp.v = static_cast<const __nv_bfloat16*>(v);
    dp.o = static_cast<__nv_bfloat16*>(o);
    dp.lse = lse;
    dp.BH = static_cast<int>(BH);
    dp.Tk = Tk;
    dp.n_splits = splits;
    dp.keys_per_split = static_cast<int>((static_cast<long long>(Tk) + splits - 1) / splits);
    dp.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    if (splits > 1) {
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      dp.o_part = reinterpret_cast<float*>(ws);
      dp.lse_part = reinterpret_cast<float*>(
          ws + round_up256(static_cast<size_t>(splits) * BH * d * 4));
    }
    if (BH * splits > INT32_MAX) return FA_ERR_INVALID_ARG;
    const cudaError_t e = fa::launch_decode(dp, d, static_cast<unsigned>(sms) * 8u,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
  }
  if (Tq <= fa::kDecMultiMaxRows) {
    // Two query rows per head: two CUDA-core warps per row, the four warps sharing every
    // K/V chunk (a 128-row tensor tile would be nearly all padding).
    fa::DecodeParams dp{};
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.k = static_cast<const __nv_bfloat16*>(k);
    dp.v = static_cast<const __nv_bfloat16*>(v);
    dp.o = static_cast<__nv_bfloat16*>(o);
    dp.lse = lse;
    dp.BH = static_cast<int>(BH);
    dp.Tk = Tk;
    dp.Tq = Tq;
    dp.causal = causal ? 1 : 0;
    dp.n_splits = splits;
    dp.keys_per_split = static_cast<int>((static_cast<long long>(Tk) + splits - 1) / splits);
    dp.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    if (splits > 1) {
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      dp.o_part = reinterpret_cast<float*>(ws);
      dp.lse_part = reinterpret_cast<float*>(
          ws + round_up256(static_cast<size_t>(splits) * BH * Tq * d * 4));
    }
    if (BH * splits > INT32_MAX) return FA_ERR_INVALID_ARG;
    const cudaError_t e = fa::launch_decode_multi(dp, d,
                                                  static_cast<unsigned>(sms) * 8u,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
  }
  GenArgs g{q, k, v, o, lse, nullptr, 1, B, H, Tq, Tk, d, causal, scale, splits, workspace,
            workspace_bytes, stream, nullptr, 0ull};
  return launch_general(g, sms);
}

int fa_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                        const unsigned char* block_mask, int mask_heads, int B, int H, int T,
                        int d, int causal, float scale, void* stream) {
  int st = validate_common(q, k, v, o, lse, B, H, T, T, d, scale);
  if (st != FA_OK) return st;
  if (!block_mask) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (mask_heads != 1 && mask_heads != BH) return FA_ERR_INVALID_ARG;
  int dev = -1, sms = 0;
  st = check_device(&dev, &sms);
  if (st != FA_OK) return st;
  GenArgs g{q, k, v, o, lse, block_mask, mask_heads, B, H, T, T, d, causal, scale, 1, nullptr,
            0, stream, nullptr, 0ull};
  return launch_general(g, sms);
}

}  // extern "C"
