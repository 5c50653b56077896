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
// In a chunk, a key is handled by G = D/32 lanes, each owning 32 of its dimensions (read
// from shared memory in a per-lane rotated column order, so that the eight lanes of a
// quarter-warp, which read eight different rows, hit eight different bank groups): the
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
  // Several query rows (fa_decode_multi_kernel): q, o are [BH][Tq][D], lse [BH][Tq], the
  // partial rows [n_splits][BH·Tq][D]; query i sees key j iff j ≤ i + Tk − Tq when causal.
  int Tq;
  int causal;
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

// Column rotation of a lane (0…3): distinct for the lanes of a quarter-warp that own the
// same bank group (D = 64: four keys × two halves; D = 128: two keys × four quarters, the
// quarters g and g + 2 sharing bank groups).
template <int D>
__device__ __forceinline__ int dec_rot(int lane) {
  if constexpr (D == 64) return (lane >> 1) & 3;
  else return ((lane & 3) >> 1) + 2 * ((lane >> 2) & 1);
}

// x[c] ← x[(c − r) mod 4] for the 8-float blocks c: a lane whose block c holds column
// 4g + (c + r) mod 4 ends with block c holding column 4g + c.
__device__ __forceinline__ void dec_unrotate(float (&x)[32], int r) {
  if (r & 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float t = x[24 + e];
      x[24 + e] = x[16 + e]; x[16 + e] = x[8 + e]; x[8 + e] = x[e]; x[e] = t;
    }
  }
  if (r & 2) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float t = x[e]; x[e] = x[16 + e]; x[16 + e] = t;
      t = x[8 + e]; x[8 + e] = x[24 + e]; x[24 + e] = t;
    }
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
    // this lane's c-th 16-byte column of a key row, in the rotated order of dec_rot
    const int rot = dec_rot<D>(lane);
    int coff[4];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) coff[c4] = (4 * g + ((c4 + rot) & 3)) * 16;
    float q[32];
    {
      const uint8_t* qr = reinterpret_cast<const uint8_t*>(p.q + static_cast<size_t>(bh) * D);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(qr + coff[c4])), q + 8 * c4);
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
      const uint8_t* kr = ring + st * 2 * kChunk + grp * kRow;
      uint4 kw[4], vw[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        kw[c4] = *reinterpret_cast<const uint4*>(kr + coff[c4]);
        vw[c4] = *reinterpret_cast<const uint4*>(kr + kChunk + coff[c4]);
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
    dec_unrotate(o, rot);
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

// A few query rows of a head against its cached keys, on the CUDA cores (used for Tq = 2). A
// query row costs the same per key as in fa_decode_kernel: a dot product and a scaled add,
// far below the tensor-core ridge, and a 128-row tensor tile would be nearly all padding.
// The four compute warps share every K/V chunk the producer brings in: warp w owns query
// row w / KP and the passes p ≡ w (mod KP) of each chunk, a pass being 32 / G keys, one per
// lane group. So the head's keys are read from memory once for the CTA's 4 / KP rows. (The
// arithmetic grows with the rows while the bytes do not: from three rows on, the one-tile
// tensor-core kernel is the faster way.)
//
// Shared-memory reads: a lane group's G lanes read a key row (2·D bytes) as 16-byte
// columns, lane g owning columns 4g…4g+3 (dimensions 32g…32g+31). The eight lanes of a
// quarter-warp read different rows, and every 128 bytes of a row span the 32 banks once, so
// reading the same column of different rows would conflict four ways. Each lane therefore
// walks its four columns in a rotated order, starting at column 4g + rot (rot fixed per
// lane, dec_rot), which gives the quarter-warp eight different bank groups; its query and
// output registers are held in the same rotated order and put back in place at the end.
//
// Each lane group keeps its own online-softmax state per row (the recurrence of step ② of
// "手写 FlashAttention", with the lazy rescale); at the end a warp merges its lane groups,
// the key parts of a row group are merged through shared memory, and the row is written:
// the bf16 row and LSE when the keys are not split, otherwise the range's fp32 row and LSE
// for fa_fwd_combine_kernel. Rows see keys up to their bottom-right causal limit.
constexpr int kDecMultiCtasPerSm = 2;

template <int D, int KP>
__global__ void __launch_bounds__(kDecBlock, kDecMultiCtasPerSm)
    fa_decode_multi_kernel(const DecodeParams p) {
  constexpr int QW = 1;                        // query rows per warp
  constexpr int G = D / 32;                    // lanes per key
  constexpr int kKeys = dec_chunk_keys<D>();   // keys per chunk
  constexpr int kRow = D * 2;
  constexpr int kChunk = kKeys * kRow;
  constexpr int kWarps = kDecThreads / 32;
  constexpr int kKPW = 32 / G;                 // keys a warp covers per pass
  constexpr int kPasses = kKeys / kKPW;
  constexpr int kGroups = kWarps / KP;         // row groups
  constexpr int kQB = kGroups * QW;            // query rows per CTA
  static_assert(kWarps % KP == 0 && kPasses % KP == 0, "key parts divide the passes");
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kDecStages], empty[kDecStages];
  __shared__ uint32_t abort_flag;
  // key parts 1…KP−1 of each row: merged state for the part-0 warp
  __shared__ float xm[KP > 1 ? kQB * (KP - 1) : 1], xl[KP > 1 ? kQB * (KP - 1) : 1];
  __shared__ __align__(16) float xo[KP > 1 ? kQB * (KP - 1) : 1][KP > 1 ? D : 1];
  pdl_wait();
  pdl_launch_dependents();
  // query blocks of one key range are neighbours in launch order (they read the same keys)
  const int n_qblk = (p.Tq + kQB - 1) / kQB;
  const int qblk = blockIdx.x % n_qblk;
  const int rest = blockIdx.x / n_qblk;
  const int bh = rest % p.BH;
  const int split = rest / p.BH;
  const int kb = split * p.keys_per_split;
  const int ke = min(p.Tk, kb + p.keys_per_split);
  const int n_chunks = ke > kb ? (ke - kb + kKeys - 1) / kKeys : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < kDecStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kWarps);
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
    const WaitCtl drain = drain_ctl(0);
    for (int x = c > kDecStages ? c - kDecStages : 0; x < c; ++x)
      mbar_wait_warp(&full[x % kDecStages], (x / kDecStages) & 1, drain);
    return;
  }
  // ---------------------------------------------------------------- compute
  const int g = lane % G;       // which 32 dimensions
  const int kgrp = lane / G;    // which key of a pass
  const int rot = dec_rot<D>(lane);
  const int rg = warp / KP, kpart = warp % KP;
  // byte offset of this lane's c-th column in a key row (rotated order)
  int coff[4];
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) coff[c4] = (4 * g + ((c4 + rot) & 3)) * 16;
  int qi[QW], lim[QW];
  float q[QW][32], o[QW][32], m[QW], l[QW];
#pragma unroll
  for (int r = 0; r < QW; ++r) {
    qi[r] = qblk * kQB + rg * QW + r;
    const bool valid = qi[r] < p.Tq;
    // keys this row may see: all, or (bottom-right causal) up to key qi + Tk − Tq
    lim[r] = !valid ? 0 : (p.causal ? qi[r] + p.Tk - p.Tq + 1 : p.Tk);
    const uint8_t* qrow = reinterpret_cast<const uint8_t*>(
        p.q + (static_cast<size_t>(bh) * p.Tq + (valid ? qi[r] : 0)) * D);
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      if (valid) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(qrow + coff[c4])), q[r] + 8 * c4);
      else {
#pragma unroll
        for (int e = 0; e < 8; ++e) q[r][8 * c4 + e] = 0.f;
      }
    }
#pragma unroll
    for (int c4 = 0; c4 < 32; ++c4) {
      q[r][c4] *= p.scale_log2;
      o[r][c4] = 0.f;
    }
    m[r] = -INFINITY;
    l[r] = 0.f;
  }
  for (int c = 0; c < n_chunks; ++c) {
    const int st = c % kDecStages;
    if (!mbar_wait_warp(&full[st], (c / kDecStages) & 1, wc)) break;
    const uint8_t* kbase = ring + st * 2 * kChunk;
#pragma unroll 2
    for (int pp = kpart; pp < kPasses; pp += KP) {
      const int kk = pp * kKPW + kgrp;             // key of the chunk
      const int key = kb + c * kKeys + kk;
      uint4 kw[4], vw[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        kw[c4] = *reinterpret_cast<const uint4*>(kbase + kk * kRow + coff[c4]);
        vw[c4] = *reinterpret_cast<const uint4*>(kbase + kChunk + kk * kRow + coff[c4]);
      }
      float sc[QW];
#pragma unroll
      for (int r = 0; r < QW; ++r) {
        float part[4];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float kf[8];
          bf16x8_to_f32(kw[c4], kf);
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) a = fmaf(kf[e], q[r][8 * c4 + e], a);
          part[c4] = a;
        }
        float a = (part[0] + part[1]) + (part[2] + part[3]);
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        sc[r] = a;
      }
      if (key >= ke) continue;  // (rows past the range were not copied: stale bytes, unused)
#pragma unroll
      for (int r = 0; r < QW; ++r) {
        if (key >= lim[r]) continue;
        if (sc[r] > m[r] + kDecTau) {  // the first key, or a max that jumped
          const float alpha = ex2_approx(m[r] - sc[r]);  // 0 while m = −∞
          l[r] *= alpha;
#pragma unroll
          for (int c4 = 0; c4 < 32; ++c4) o[r][c4] *= alpha;
          m[r] = sc[r];
        }
        const float pj = ex2_approx(sc[r] - m[r]);
        l[r] += pj;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float vf[8];
          bf16x8_to_f32(vw[c4], vf);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[r][8 * c4 + e] = fmaf(pj, vf[e], o[r][8 * c4 + e]);
        }
      }
    }
    // this warp's passes of the chunk are done: the producer may refill the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  const bool failed = abort_flag != 0u;
  const float nan = __uint_as_float(0x7FC00000u);
  float mw[QW], lw[QW];
#pragma unroll
  for (int r = 0; r < QW; ++r) {
    // merge the warp's lane groups (lanes with the same g): rescale to their max, then add
    dec_unrotate(o[r], rot);
    mw[r] = m[r];
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) mw[r] = fmaxf(mw[r], __shfl_xor_sync(0xffffffffu, mw[r], off));
    const float f = (m[r] == -INFINITY) ? 0.f : ex2_approx(m[r] - mw[r]);
    lw[r] = l[r] * f;
#pragma unroll
    for (int off = 16; off >= G; off >>= 1) lw[r] += __shfl_xor_sync(0xffffffffu, lw[r], off);
#pragma unroll
    for (int c4 = 0; c4 < 32; ++c4) {
      float x = o[r][c4] * f;
#pragma unroll
      for (int off = 16; off >= G; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      o[r][c4] = x;
    }
  }
  if constexpr (KP > 1) {
    // the other key parts hand their rows to part 0 (named barrier: compute warps only)
    if (kpart > 0 && lane < G) {
#pragma unroll
      for (int r = 0; r < QW; ++r) {
        const int slot = (rg * QW + r) * (KP - 1) + kpart - 1;
        if (lane == 0) {
          xm[slot] = mw[r];
          xl[slot] = lw[r];
        }
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) xo[slot][g * 32 + c4] = o[r][c4];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory");
    if (kpart > 0) return;
#pragma unroll
    for (int r = 0; r < QW; ++r) {
      float M = mw[r];
#pragma unroll
      for (int x = 0; x < KP - 1; ++x) M = fmaxf(M, xm[(rg * QW + r) * (KP - 1) + x]);
      const float f0 = (mw[r] == -INFINITY) ? 0.f : ex2_approx(mw[r] - M);
      float L = lw[r] * f0;
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) o[r][c4] *= f0;
#pragma unroll
      for (int x = 0; x < KP - 1; ++x) {
        const int slot = (rg * QW + r) * (KP - 1) + x;
        const float fx = (xm[slot] == -INFINITY) ? 0.f : ex2_approx(xm[slot] - M);
        L = fmaf(fx, xl[slot], L);
#pragma unroll
        for (int c4 = 0; c4 < 32; ++c4) o[r][c4] = fmaf(fx, xo[slot][g * 32 + c4], o[r][c4]);
      }
      mw[r] = M;
      lw[r] = L;
    }
  }
#pragma unroll
  for (int r = 0; r < QW; ++r) {
    if (qi[r] >= p.Tq || lane >= G) continue;
    const bool empty_row = !(lw[r] > 0.f);
    const float inv_l = empty_row ? 0.f : 1.f / lw[r];
    float lse_v = empty_row ? -INFINITY : (mw[r] + log2f(lw[r])) * 0.69314718055994530942f;
    if (failed) lse_v = nan;
    const size_t row = static_cast<size_t>(bh) * p.Tq + qi[r];
    if (p.n_splits == 1) {
      uint32_t* orow = reinterpret_cast<uint32_t*>(p.o + row * D + g * 32);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4)
        orow[c4] = failed ? 0x7FC07FC0u : pack_bf16x2(o[r][2 * c4] * inv_l, o[r][2 * c4 + 1] * inv_l);
      if (lane == 0) p.lse[row] = lse_v;
    } else {
      const size_t prow = static_cast<size_t>(split) * p.BH * p.Tq + row;
      float* op = p.o_part + prow * D + g * 32;
#pragma unroll
      for (int c4 = 0; c4 < 32; ++c4) op[c4] = failed ? nan : o[r][c4] * inv_l;
      if (lane == 0) p.lse_part[prow] = lse_v;
    }
  }
}

}  // namespace fa
