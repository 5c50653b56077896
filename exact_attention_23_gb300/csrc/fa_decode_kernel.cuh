// Decode: one query row per (batch, head) against Tk cached keys, on the CUDA cores.
//
// With a single query the work is a dot product and a scaled add per cached K/V row: two
// FLOPs per byte read, far below any tensor-core ridge, so the kernel is a streaming
// kernel whose job is to keep enough bytes in flight. A key is handled by G = D/32 lanes,
// each owning 32 of its dimensions: the lane's partial dot product is completed with
// log2(G) shuffles, and its 32 output accumulators take the key's contribution. Each lane
// group keeps its own online-softmax state — running max m (base 2), running sum l,
// accumulator o — exactly the recurrence of step ② of "手写 FlashAttention" (Hand-written
// FlashAttention), with the lazy rescale (o and l keep a stale max until a score exceeds it
// by τ). The K and V rows of kDecKeys keys are requested together before any is used, so a
// round trip to memory serves several keys. At the end the states of a warp, then of the
// CTA's warps, are merged (rescaled to the larger max, added); the CTA writes its key
// range's result: the final bf16 row and LSE when the keys are not split, otherwise the
// normalised fp32 row and LSE of the range, which fa_fwd_combine_kernel merges.
#pragma once

#include "sm103.cuh"

namespace fa {

struct DecodeParams {
  const __nv_bfloat16* q;  // [BH][D]: the one query row of each head
  const __nv_bfloat16* k;  // [BH][Tk][D]
  const __nv_bfloat16* v;  // [BH][Tk][D]
  __nv_bfloat16* o;        // [BH][D] (n_splits == 1)
  float* lse;              // [BH]    (n_splits == 1)
  float* o_part;           // [n_splits][BH][D] fp32 (n_splits > 1)
  float* lse_part;         // [n_splits][BH]        (n_splits > 1)
  int BH;
  int Tk;
  int n_splits;
  int keys_per_split;
  float scale_log2;        // scale · log2(e)
};

constexpr int kDecThreads = 128;
constexpr int kDecKeys = 2;      // keys whose rows each lane requests before using them
constexpr int kDecCtasPerSm = 3;
constexpr float kDecTau = 8.0f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(u[e] << 16);
    f[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
  }
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm)
    fa_decode_kernel(const DecodeParams p) {
  constexpr int G = D / 32;                     // lanes per key
  constexpr int kGroups = kDecThreads / G;      // keys in flight per CTA step (× kDecKeys)
  constexpr int kWarps = kDecThreads / 32;
  __shared__ float wm[kWarps], wl[kWarps];
  __shared__ __align__(16) float wo[kWarps][D];
  // Launched as a programmatic dependent: the previous kernel on the stream (possibly the
  // last merge, which reads o_part) must be complete before anything is read or written.
  pdl_wait();
  pdl_launch_dependents();
  const int bh = blockIdx.x % p.BH;
  const int split = blockIdx.x / p.BH;
  const int kb = split * p.keys_per_split;
  const int ke = min(p.Tk, kb + p.keys_per_split);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane % G;                        // which 32 dimensions
  const int grp = static_cast<int>(threadIdx.x) / G;  // which key of a step

  float q[32];
  {
    const uint4* qr = reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(bh) * D + g * 32);
#pragma unroll
    for (int c = 0; c < 4; ++c) bf16x8_to_f32(__ldg(qr + c), q + 8 * c);
#pragma unroll
    for (int c = 0; c < 32; ++c) q[c] *= p.scale_log2;
  }
  float m = -INFINITY, l = 0.f;
  float o[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) o[c] = 0.f;
  const __nv_bfloat16* kh = p.k + static_cast<size_t>(bh) * p.Tk * D + g * 32;
  const __nv_bfloat16* vh = p.v + static_cast<size_t>(bh) * p.Tk * D + g * 32;

  // Every lane runs the same number of steps (the shuffles need the whole warp); keys past
  // the range are loaded from row kb (in bounds) and weighted 0.
  for (int base = kb; base < ke; base += kGroups * kDecKeys) {
    uint4 kw[kDecKeys][4], vw[kDecKeys][4];
    bool live[kDecKeys];
#pragma unroll
    for (int t = 0; t < kDecKeys; ++t) {
      const int j = base + t * kGroups + grp;
      live[t] = j < ke;
      const size_t row = static_cast<size_t>(live[t] ? j : kb) * D;
      const uint4* kr = reinterpret_cast<const uint4*>(kh + row);
      const uint4* vr = reinterpret_cast<const uint4*>(vh + row);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        kw[t][c] = __ldg(kr + c);
        vw[t][c] = __ldg(vr + c);
      }
    }
#pragma unroll
    for (int t = 0; t < kDecKeys; ++t) {
      float sc = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float kf[8];
        bf16x8_to_f32(kw[t][c], kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc = fmaf(kf[e], q[8 * c + e], sc);
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      if (!live[t]) continue;
      if (sc > m + kDecTau) {  // the first key, or a max that jumped: move the reference
        const float alpha = ex2_approx(m - sc);  // 0 while m = −∞
        l *= alpha;
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] *= alpha;
        m = sc;
      }
      const float pj = ex2_approx(sc - m);
      l += pj;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float vf[8];
        bf16x8_to_f32(vw[t][c], vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[8 * c + e] = fmaf(pj, vf[e], o[8 * c + e]);
      }
    }
  }

  // Merge the warp's key groups (lanes with the same g): rescale to their max, then add.
  float mw = m;
#pragma unroll
  for (int off = 16; off >= G; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
  const float f = (m == -INFINITY) ? 0.f : ex2_approx(m - mw);
  l *= f;
#pragma unroll
  for (int off = 16; off >= G; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    float x = o[c] * f;
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    o[c] = x;
  }
  if (lane < G) {
    if (lane == 0) {
      wm[warp] = mw;
      wl[warp] = l;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) wo[warp][g * 32 + c] = o[c];
  }
  __syncthreads();

  // Merge the warps: thread c owns output column c.
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w]);
  float L = 0.f;
  float wgt[kWarps];
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    wgt[w] = (wm[w] == -INFINITY) ? 0.f : ex2_approx(wm[w] - M);
    L += wgt[w] * wl[w];
  }
  const bool empty = !(L > 0.f);
  const float inv_l = empty ? 0.f : 1.f / L;
  const float lse_v = empty ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
  for (int c = threadIdx.x; c < D; c += kDecThreads) {
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) x = fmaf(wgt[w], wo[w][c], x);
    x *= inv_l;
    if (p.n_splits == 1) {
      p.o[static_cast<size_t>(bh) * D + c] = __float2bfloat16_rn(x);
    } else {
      p.o_part[(static_cast<size_t>(split) * p.BH + bh) * D + c] = x;
    }
  }
  if (threadIdx.x == 0) {
    if (p.n_splits == 1) p.lse[bh] = lse_v;
    else p.lse_part[static_cast<size_t>(split) * p.BH + bh] = lse_v;
  }
}

}  // namespace fa
