// Decode: one query row per (batch, head) against Tk cached keys, on the CUDA cores.
//
// With a single query the work is a dot product and a scaled add per cached K/V row: two
// FLOPs per byte read, far below any tensor-core ridge, so the kernel is a streaming
// kernel whose job is to keep enough bytes in flight. Each CTA owns one key range of one
// head. A producer warp streams the range's K and V rows through a ring of kDecStages
// shared-memory stages with bulk copies (contiguous chunks of kKeys rows, completed on an
// mbarrier), so the copies stay in flight while the four compute warps work: a compute
// warp never waits for a round trip it could have overlapped.
//
// In a chunk, a key is handled by G = D/32 lanes, each owning 32 of its dimensions: the
// lane's partial dot product is completed with log2(G) shuffles, and its 32 output
// accumulators take the key's contribution. Each lane group keeps its own online-softmax
// state — running max m (base 2), running sum l, accumulator o — exactly the recurrence of
// step ② of "手写 FlashAttention" (Hand-written FlashAttention), with the lazy rescale (o and
// l keep a stale max until a score exceeds it by τ). At the end the states of a warp, then
// of the CTA's warps, are merged (rescaled to the larger max, added); the CTA writes its
// key range's result: the final bf16 row and LSE when the keys are not split, otherwise the
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

constexpr int kDecThreads = 128;             // compute threads (4 warps)
constexpr int kDecBlock = kDecThreads + 32;  // + the producer warp
constexpr int kDecStages = 4;                // K/V chunks in flight per CTA
constexpr int kDecCtasPerSm = 3;
constexpr float kDecTau = 8.0f;

// Keys per chunk (one per lane group) and the ring's bytes: kDecStages × (K chunk + V chunk),
// 64 KB at either head dim.
template <int D>
__host__ __device__ constexpr int dec_chunk_keys() { return kDecThreads / (D / 32); }
template <int D>
__host__ __device__ constexpr int dec_smem_bytes() { return kDecStages * 2 * dec_chunk_keys<D>() * D * 2; }

__device__ __forceinline__ void bf16x8_to_f32(const uint4& w, float* f) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    f[2 * e] = __uint_as_float(u[e] << 16);
    f[2 * e + 1] = __uint_as_float(u[e] & 0xFFFF0000u);
  }
}

template <int D>
__global__ void __launch_bounds__(kDecBlock, kDecCtasPerSm)
    fa_decode_kernel(const DecodeParams p) {
  constexpr int G = D / 32;                    // lanes per key
  constexpr int kKeys = dec_chunk_keys<D>();   // keys per chunk
  constexpr int kRow = D * 2;                  // bytes of one K or V row
  constexpr int kChunk = kKeys * kRow;         // bytes of one K (or V) chunk
  constexpr int kWarps = kDecThreads / 32;     // compute warps; warp kWarps is the producer
  extern __shared__ __align__(128) uint8_t ring[];  // stage s: K chunk, then V chunk
  __shared__ uint64_t full[kDecStages], empty[kDecStages];
  __shared__ uint32_t abort_flag;
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
  const int n_chunks = ke > kb ? (ke - kb + kKeys - 1) / kKeys : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, nullptr, 2000000000ull};

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    const uint8_t* kg = reinterpret_cast<const uint8_t*>(p.k + static_cast<size_t>(bh) * p.Tk * D);
    const uint8_t* vg = reinterpret_cast<const uint8_t*>(p.v + static_cast<size_t>(bh) * p.Tk * D);
    int c = 0;
    for (; c < n_chunks; ++c) {
      const int st = c % kDecStages;
      if (c >= kDecStages && !mbar_wait_warp(&empty[st], ((c / kDecStages) - 1) & 1, wc)) break;
      const int k0 = kb + c * kKeys;
      const uint32_t bytes = static_cast<uint32_t>(min(kKeys, ke - k0) * kRow);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[st], 2 * bytes);
        bulk_load(ring + st * 2 * kChunk, kg + static_cast<size_t>(k0) * kRow, bytes, &full[st]);
        bulk_load(ring + st * 2 * kChunk + kChunk, vg + static_cast<size_t>(k0) * kRow, bytes,
                  &full[st]);
      }
      __syncwarp();
    }
    // Every copy issued must have landed before the CTA may exit (the compute warps have
    // consumed them all unless a wait gave up).
    const WaitCtl drain = drain_ctl(0);
    for (int x = c > kDecStages ? c - kDecStages : 0; x < c; ++x)
      mbar_wait_warp(&full[x % kDecStages], (x / kDecStages) & 1, drain);
  } else {
    // ---------------------------------------------------------------- compute
    const int g = lane % G;                               // which 32 dimensions
    const int grp = static_cast<int>(threadIdx.x) / G;    // which key of a chunk
    float q[32];
    {
      const uint4* qr = reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(bh) * D + g * 32);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) bf16x8_to_f32(__ldg(qr + c4), q + 8 * c4);
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) q[c4] *= p.scale_log2;
    }
    float m = -INFINITY, l = 0.f;
    float o[32];
#pragma unroll
    for (int c4 = 0; c4 < 32; ++c4) o[c4] = 0.f;
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % kDecStages;
      if (!mbar_wait_warp(&full[st], (c / kDecStages) & 1, wc)) break;
      const bool live = kb + c * kKeys + grp < ke;
      const uint4* kr = reinterpret_cast<const uint4*>(ring + st * 2 * kChunk + grp * kRow + g * 64);
      const uint4* vr = reinterpret_cast<const uint4*>(ring + st * 2 * kChunk + kChunk +
                                                       grp * kRow + g * 64);
      uint4 kw[4], vw[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        kw[c4] = kr[c4];
        vw[c4] = vr[c4];
      }
      // The chunk is in registers: the producer may refill the stage.
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      float sc = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float kf[8];
        bf16x8_to_f32(kw[c4], kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) sc = fmaf(kf[e], q[8 * c4 + e], sc);
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      if (!live) continue;  // (rows past the range were not copied: stale bytes, unused)
      if (sc > m + kDecTau) {  // the first key, or a max that jumped: move the reference
        const float alpha = ex2_approx(m - sc);  // 0 while m = −∞
        l *= alpha;
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) o[c4] *= alpha;
        m = sc;
      }
      const float pj = ex2_approx(sc - m);
      l += pj;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float vf[8];
        bf16x8_to_f32(vw[c4], vf);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[8 * c4 + e] = fmaf(pj, vf[e], o[8 * c4 + e]);
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
    for (int c4 = 0; c4 < 32; ++c4) {
      float x = o[c4] * f;
#pragma unroll
      for (int off = 16; off >= G; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      o[c4] = x;
    }
    if (lane < G) {
      if (lane == 0) {
        wm[warp] = mw;
        wl[warp] = l;
      }
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) wo[warp][g * 32 + c4] = o[c4];
    }
  }
  __syncthreads();
  if (warp == kWarps) return;

  // Merge the warps: thread c owns output column c. A CTA whose waits gave up writes NaN.
  const bool failed = abort_flag != 0u;
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
  const bool empty_row = !(L > 0.f);
  const float inv_l = empty_row ? 0.f : 1.f / L;
  const float nan = __uint_as_float(0x7FC00000u);
  float lse_v = empty_row ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f;
  if (failed) lse_v = nan;
  for (int c = threadIdx.x; c < D; c += kDecThreads) {
    float x = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) x = fmaf(wgt[w], wo[w][c], x);
    x = failed ? nan : x * inv_l;
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
