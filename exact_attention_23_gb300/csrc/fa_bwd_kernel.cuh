// Exact attention backward for GB300 (sm_103a): the gradients dQ, dK, dV of
// O = softmax(scale·QKᵀ [+causal mask])·V for an upstream gradient dO.
//
// The forward keeps only the row logsumexp LSE; the backward recomputes the scores and
// probabilities block by block from it instead of storing the T×T matrix, as step ④ of
// "手写 FlashAttention" (Hand-written FlashAttention, learn-llm.fim.ai ch. 19) and §2.2 of
// "FlashAttention 核心思路解析" (FlashAttention core ideas, ijyty.com: recompute per block,
// sum the per-block query gradients into the global gradient with atomic adds) describe.
// With D_i = Σ_c dO_ic·O_ic, for a query tile i and key tile j:
//
//   Pᵀ  = exp2(log2(e)·scale·K_j·Q_iᵀ − log2(e)·LSE_i)   (keys on TMEM lanes)
//   dPᵀ = V_j·dO_iᵀ
//   dSᵀ = Pᵀ ∘ (dPᵀ − D_i)
//   dV_j += Pᵀ·dO_i      dK_j += dSᵀ·Q_i      dQ_i += dS·K_j   (dK, dQ × scale at the end)
//
// Three kernels per call:
//   fa_bwd_prep_kernel   D_i, log2(e)·LSE_i (+∞ on padding rows, so their P is 0) and a
//                        zeroed fp32 dQ accumulator, all in the caller's workspace;
//   fa_bwd_main_kernel   one CTA per (128-key tile j, batch·head), walking the query tiles
//                        the mask leaves visible; dK_j, dV_j stay in TMEM for the whole walk,
//                        dQ_i partials are added to the accumulator;
//   fa_bwd_dq_kernel     accumulator × scale → bf16 dQ.
//
// Main kernel: kCWG compute warpgroups (4 at d = 64: 23 warps, 736 threads; 2 at d = 128:
// 16 warps, 512 threads), then:
//   warps 0 .. 4·kCWG−1   compute: warpgroup g owns query columns 32·g .. 32·g+31 of each
//                         tile (thread = key row); no exchange between warpgroups is needed,
//                         since P comes from the saved LSE, column by column
//   next 4 warps          dQ drain: TMEM → registers → shared memory → bulk reduce-adds
//                         into the fp32 accumulator by the TMA engine
//   next warp             score issuer: Sᵀ and dPᵀ MMAs (one elected thread); TMEM owner
//   next warp             gradient issuer: dV, dK and dQ MMAs (one elected thread); at
//                         d = 128 dV and dK only
//   next warp             TMA producer
//   last warp (d = 128)   dQ issuer: the dQᵀ MMAs, from the fourth sub-partition (measured
//                         4 % faster there; at d = 64 a separate dQ issuer was 2 % slower)
// (More compute warps hide more of the latency of each tile's chain of TMEM loads and
// stores; at d = 64 four warpgroups of 32 columns measured 4 % faster than two of 64.)
// Two issuers, because MMAs into different accumulators are not ordered with one another
// and a single issuer blocked on one barrier would hold back independent work: the score
// issuer starts Sᵀ of the next tile as soon as the compute warps have read the current
// one into registers, while the gradient issuer is still waiting for this tile's Pᵀ/dSᵀ.
// Pᵀ goes to tensor memory (bf16 pairs, the A operand of the dV MMA). dSᵀ is written to
// shared memory as bf16 in the 128-byte-swizzled layout a TMA load would produce
// ([key row][64 query columns] boxes, double-buffered). The same bytes serve as the
// K-major A operand of dK (rows = keys) and the MN-major A operand of dQ (queries on M),
// so no transpose is ever materialised.
// Tensor memory (D = 64): [0,128) Sᵀ, [128,256) dPᵀ, [256,320) dV, [320,384) dK,
// [384,448) dQ, [448,512) Pᵀ (bf16 pairs).
#pragma once

#include "sm103.cuh"

// Timeline hooks: compiled out unless a tracing build defines FA_TRACE(tag, step).
#ifndef FA_TRACE
#define FA_TRACE(tag, step) ((void)0)
#endif

namespace fa {


// Tile shapes. Keys are always in 128-row tiles (the TMEM lanes of Sᵀ, dPᵀ, dV and dK).
// Query tiles have kBQ rows: 128 at d = 64; 64 at d = 128, where 128-column Sᵀ, dPᵀ, dV and
// dK would already fill the 512 TMEM columns. With 64-query tiles every product keeps
// M = 128: dQ is then made transposed, dQᵀ = Kᵀ·dSᵀ (head dims on TMEM lanes, N = 64).
template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kBQ = (D == 64) ? 128 : 64;    // query rows per tile
  // Compute warpgroups, each owning kNC query columns of a tile (32 at either head dim).
  static constexpr int kCWG = (D == 64) ? 4 : 2;  // (4 at d = 128, 16 columns each: 3 % slower)
  static constexpr int kNC = kBQ / kCWG;
  static constexpr int kComputeWarps = 4 * kCWG;
  // Warp roles after the compute warps: 4 dQ drain warps, score issuer, gradient issuer,
  // TMA producer.
  static constexpr int kDrainWarp0 = kComputeWarps;
  static constexpr int kScoreWarp = kDrainWarp0 + 4;
  static constexpr int kGradWarp = kScoreWarp + 1;
  static constexpr int kLoadWarp = kScoreWarp + 2;
  static constexpr bool kSplitQ = (D == 128);  // dQ products issued by a warp of their own
  static constexpr int kGradQWarp = kScoreWarp + 3;
  static constexpr int kThreads = (kSplitQ ? kGradQWarp + 1 : kLoadWarp + 1) * 32;
  static constexpr int kBox = 128 * 64 * 2;           // 128 rows × 64 bf16 columns = 16 KB
  static constexpr int kQBox = kBQ * 64 * 2;          // kBQ rows × 64 columns
  static constexpr int kKVTile = 128 * D * 2;         // a K or V tile
  static constexpr int kQTile = kBQ * D * 2;          // a Q or dO tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKVTile;
  static constexpr int kStages = 3;                   // (Q_i, dO_i) ring depth
  static constexpr int kStage0 = kV + kKVTile;        // stage s: Q at +0, dO at +kQTile
  static constexpr int kStageBytes = 2 * kQTile;
  static constexpr int kDS = kStage0 + kStages * kStageBytes;  // dSᵀ: 2 buffers
  static constexpr int kDSBytes = 128 * kBQ * 2;      // [128 keys][kBQ queries] bf16, 64-col boxes
  static constexpr int kVecBytes = 2 * kBQ * 4;       // per stage: −lse2[kBQ] then D[kBQ]
  static constexpr int kVec = kDS + 2 * kDSBytes;
  // Each dQ drain warp stages 16 of its TMEM columns for its 32 lanes (2 KB) for a bulk
  // reduce-add, two buffers per warp.
  static constexpr int kDQChunk = 32 * 16 * 4;
  static constexpr int kDQStage = kVec + kStages * kVecBytes;
  static constexpr int kBar = kDQStage + 4 * 2 * kDQChunk;
  static constexpr int kSmemBytes = kBar + 256 + 1024;  // barriers + 1 KB alignment slack
  // Tensor memory: Sᵀ, dPᵀ (kBQ columns each), dV, dK (D each), dQ (D columns at d = 64,
  // dQᵀ with kBQ columns at d = 128), Pᵀ as bf16 pairs (kBQ/2 columns).
  static constexpr uint32_t kColS = 0, kColDP = kBQ, kColDV = 2 * kBQ, kColDK = 2 * kBQ + D;
  static constexpr uint32_t kColDQ = 2 * kBQ + 2 * D;
  static constexpr uint32_t kColP = kColDQ + ((D == 64) ? D : kBQ);
  static_assert(kColP + kBQ / 2 <= 512, "tensor memory");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct BwdBars {
  uint64_t kv_full;     // K_j, V_j landed
  uint64_t q_full[3];   // Q_i, dO_i, lse2_i, D_i landed in a stage
  uint64_t q_empty[3];  // both issuers' MMAs reading that stage are done (2 arrivals)
  uint64_t s_full;      // Sᵀ in TMEM
  uint64_t s_free;      // Sᵀ read into registers (8 compute warps)
  uint64_t dp_full;     // dPᵀ in TMEM
  uint64_t dp_free;     // dPᵀ read into registers (8 compute warps)
  uint64_t p_full;      // Pᵀ stored in TMEM (8 compute warps)
  uint64_t p_free;      // dV MMA done with Pᵀ
  uint64_t ds_full[2];  // dSᵀ buffer in shared memory (8 compute warps)
  uint64_t ds_free[2];  // dK and dQ MMAs done with that buffer
  uint64_t dq_full;     // a dQ partial in TMEM
  uint64_t dq_free;     // drained (4 drain warps)
  uint64_t score_done;  // every MMA of the score issuer done
  uint64_t grad_done;   // every MMA of the gradient issuer done: dK, dV final
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");

struct BwdParams {
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* lse2;   // [BH][T_pad] −log2(e)·LSE, −∞ on padding rows
  const float* dvec;   // [BH][T_pad] D_i, 0 on padding rows
  float* dq_acc;       // fp32 dQ accumulator (unscaled), layout of dq_acc_offset
  int* status;
  int T;
  int T_pad;           // ceil(T / 128) · 128
  int BH;
  int n_qt;            // T_pad / kBQ query tiles
  int n_kt;            // T_pad / 128 key tiles
  int head_group;      // heads whose units are interleaved (see the unit order)
  float scale;
  float scale_log2;    // scale · log2(e)
  uint64_t timeout_ns;
  uint32_t flags;
};

constexpr uint32_t kBwdFlagStarveQ = 1u;  // FA_FLAG_TEST_STARVE_Q

// dQ accumulator layouts.
// d = 64 (thread = query row r of a 128-row tile): [bh][tile][r/32][d/4][32 rows][4 columns],
//   so the 32 rows of one drain warp and 16 consecutive columns are 2 KB in one piece (one
//   bulk reduce-add); dq_acc_offset(bh, i, n_qt, c4, r, d) is query row r, columns
//   4·c4 .. 4·c4+3.
// d = 128 (dQᵀ: thread = head dim c of a 64-query tile): [bh][tile][c/32][16][32 dims][4 rows],
//   so the 32 dims of one drain warp and 16 consecutive query rows are 2 KB in one piece;
//   dq_acc_offset_t(bh, i, n_qt, g, c) is head dim c of query rows 4·g .. 4·g+3.
// N consecutive TMEM columns (N = 16 or a multiple of 32) of the warp's 32 lanes into r,
// with one wait for all of them.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, r);
    tmem_ld_wait();
    reg_fence16(r);
  } else {
#pragma unroll
    for (int h = 0; h < N / 32; ++h) tmem_ld32(taddr + h * 32, r + h * 32);
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < N / 32; ++h) reg_fence32(r + h * 32);
  }
}

__host__ __device__ __forceinline__ size_t dq_acc_offset(int bh, int i, int n_qt, int c4, int r,
                                                         int d) {
  return (((((size_t)bh * n_qt + i) * 4u + (unsigned)(r >> 5)) * (size_t)(d / 4) + c4) * 32u +
          (unsigned)(r & 31)) * 4u;
}
__host__ __device__ __forceinline__ size_t dq_acc_offset_t(int bh, int i, int n_qt, int g, int c) {
  return (((((size_t)bh * n_qt + i) * 4u + (unsigned)(c >> 5)) * 16u + g) * 32u +
          (unsigned)(c & 31)) * 4u;
}

// ------------------------------------------------------------------------------------
// Preprocessing: D_i = Σ_c dO_ic·O_ic, lse2_i = −log2(e)·LSE_i (negated: the main kernel adds
// it in a packed fp32x2 FMA); zero the dQ accumulator.
// D/8 consecutive lanes share a row, each reading 8 columns (16 bytes) of O and dO.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                          const __nv_bfloat16* __restrict__ dout,
                                                          const float* __restrict__ lse,
                                                          float* __restrict__ lse2,
                                                          float* __restrict__ dvec,
                                                          float* __restrict__ dq_acc, int T,
                                                          int T_pad, int BH) {
  constexpr int L = D / 8;
  pdl_wait();  // launched as a programmatic dependent (o, dO and lse may come from the previous kernel)
  pdl_launch_dependents();
  const size_t nrows = (size_t)BH * T_pad;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  // T_pad is a multiple of 128, so nrows·L is a multiple of 32 and every lane of a warp
  // runs the same number of iterations (the shuffles below need the whole warp).
  for (size_t idx = tid; idx < nrows * L; idx += stride) {
    const size_t row = idx / L;
    const int c = static_cast<int>(idx % L);
    const int bh = static_cast<int>(row / T_pad);
    const int t = static_cast<int>(row % T_pad);
    float acc = 0.f;
    if (t < T) {
      const size_t off = ((size_t)bh * T + t) * D + (size_t)c * 8;
      const uint4 a = *reinterpret_cast<const uint4*>(o + off);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + off);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
        const float2 fb2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[e]));
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
    }
#pragma unroll
    for (int w = L / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
    if (c == 0) {
      dvec[row] = (t < T) ? acc : 0.f;
      lse2[row] = (t < T) ? lse[(size_t)bh * T + t] * -1.4426950408889634f : __int_as_float(0xff800000);
    }
  }
  float4* acc4 = reinterpret_cast<float4*>(dq_acc);
  const size_t n4 = nrows * (D / 4);
  for (size_t x = tid; x < n4; x += stride) acc4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------------------------
// dQ = scale · accumulator, as bf16 rows.
// d = 64: one thread per (tile, 8 columns, row). d = 128: one thread per (64-row tile,
// group of 4 rows, 8 head dims), writing 4 rows × 8 columns.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ dq_acc,
                                                        __nv_bfloat16* __restrict__ dq, int T,
                                                        int n_qt, int BH, float scale) {
  constexpr int C8 = D / 8;
  pdl_wait();  // launched as a programmatic dependent of the main kernel (dq_acc)
  pdl_launch_dependents();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  if constexpr (D == 64) {
    const size_t total = (size_t)BH * n_qt * C8 * 128;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
      const int r = static_cast<int>(idx % 128);
      const size_t rest = idx / 128;
      const int c8 = static_cast<int>(rest % C8);
      const size_t tile = rest / C8;  // bh · n_qt + i
      const int i = static_cast<int>(tile % n_qt);
      const int bh = static_cast<int>(tile / n_qt);
      const int t = i * 128 + r;
      if (t >= T) continue;
      const float4 a = *reinterpret_cast<const float4*>(dq_acc + dq_acc_offset(bh, i, n_qt, 2 * c8, r, D));
      const float4 b = *reinterpret_cast<const float4*>(dq_acc + dq_acc_offset(bh, i, n_qt, 2 * c8 + 1, r, D));
      uint4 out;
      out.x = pack_bf16x2(a.x * scale, a.y * scale);
      out.y = pack_bf16x2(a.z * scale, a.w * scale);
      out.z = pack_bf16x2(b.x * scale, b.y * scale);
      out.w = pack_bf16x2(b.z * scale, b.w * scale);
      *reinterpret_cast<uint4*>(dq + ((size_t)bh * T + t) * D + (size_t)c8 * 8) = out;
    }
  } else {
    const size_t total = (size_t)BH * n_qt * 16 * C8;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
      const int c8 = static_cast<int>(idx % C8);
      const size_t rest = idx / C8;
      const int g = static_cast<int>(rest % 16);
      const size_t tile = rest / 16;
      const int i = static_cast<int>(tile % n_qt);
      const int bh = static_cast<int>(tile / n_qt);
      float4 col[8];  // head dims c8·8 .. c8·8+7, each holding rows 4g .. 4g+3
#pragma unroll
      for (int e = 0; e < 8; ++e)
        col[e] = *reinterpret_cast<const float4*>(dq_acc + dq_acc_offset_t(bh, i, n_qt, g, c8 * 8 + e));
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int t = i * 64 + 4 * g + rr;
        if (t >= T) break;
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 cv = col[e];
          y[e] = (rr == 0 ? cv.x : rr == 1 ? cv.y : rr == 2 ? cv.z : cv.w) * scale;
        }
        uint4 out;
        out.x = pack_bf16x2(y[0], y[1]);
        out.y = pack_bf16x2(y[2], y[3]);
        out.z = pack_bf16x2(y[4], y[5]);
        out.w = pack_bf16x2(y[6], y[7]);
        *reinterpret_cast<uint4*>(dq + ((size_t)bh * T + t) * D + (size_t)c8 * 8) = out;
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// Main kernel.
// ------------------------------------------------------------------------------------
// Stores 8 fp32 values of one row as bf16 into a 128-byte-swizzled box: 16-byte chunk
// `ch` of row `r` sits at chunk position ch ^ (r mod 8), as a TMA load would place it.
__device__ __forceinline__ void st_row_chunk_sw128(uint32_t box, int r, int ch, const float* x) {
  st_shared_v4(box + static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(ch ^ (r & 7)) << 4),
               pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
               pack_bf16x2(x[6], x[7]));
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BwdBars* bars = reinterpret_cast<BwdBars*>(sm + C::kBar);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Unit order: heads in groups of head_group, small enough that a group's Q, dO and dQ
  // accumulator stay in L2 while its CTAs run; within a group, heaviest units first (under
  // the causal mask key tile j sees the query tiles from the one holding query 128·j on),
  // all heads at one j together.
  const int per_group = p.head_group * p.n_kt;
  const int grp = blockIdx.x / per_group;
  const int within = blockIdx.x - grp * per_group;
  const int gsize = min(p.head_group, p.BH - grp * p.head_group);
  const int j = within / gsize;
  const int bh = grp * p.head_group + within % gsize;
  const int i0 = CAUSAL ? (j * 128) / C::kBQ : 0;
  const int n = p.n_qt - i0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->ds_full[s], C::kComputeWarps);
      mbar_init(&bars->ds_free[s], C::kSplitQ ? 2 : 1);  // after dK (and dQ, if split)
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, C::kComputeWarps);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, C::kComputeWarps);
    mbar_init(&bars->p_full, C::kComputeWarps);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);
    mbar_init(&bars->score_done, 1);
    mbar_init(&bars->grad_done, C::kSplitQ ? 2 : 1);
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == C::kScoreWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Launched as a programmatic dependent of the prep kernel: the set-up above overlapped its
  // tail; its outputs (D, log2e·LSE, the zeroed dQ accumulator) are read only after this.
  // (No early trigger for the dQ conversion: letting it be scheduled during this grid's
  // last wave measured 5 % slower at d = 128.)
  pdl_wait();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, p.status, p.timeout_ns};
  const WaitCtl drain_wc = drain_ctl(p.timeout_ns);
  const uint32_t sbase = smem_u32(sm);
  auto q_s = [&](int st) { return sbase + C::kStage0 + st * C::kStageBytes; };
  auto do_s = [&](int st) { return q_s(st) + C::kQTile; };
  // Operand steps: K-major, 16 columns = 32 bytes inside a 64-column box, next box `box`
  // bytes on; MN-major, 16 rows = 2 KB, boxes along M/N `box` bytes apart (leading byte
  // offset). K/V tiles and dSᵀ have 128-row boxes (16 KB); Q/dO tiles kBQ-row boxes.
  auto kmaj = [&](uint32_t base, int kk, uint32_t box) {
    return sdesc_sw128(base + (kk >> 2) * box + (kk & 3) * 32, 16, 1024);
  };
  auto mnmaj = [&](uint32_t base, int kk, uint32_t box) {
    return sdesc_sw128(base + kk * 2048, box, 1024);
  };
  // End of every role (each calls it last, so that no code is shared between warpgroups
  // that run with different register budgets). Nothing may be in flight on the tensor
  // core when TMEM is released.
  auto teardown = [&]() {
    if (warp == C::kScoreWarp) {
      mbar_wait_warp_inl(&bars->score_done, 0, drain_wc);
      mbar_wait_warp_inl(&bars->grad_done, 0, drain_wc);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::kScoreWarp) {
      tc_fence_after_sync();
      tmem_dealloc(tmem, 512);
    }
  };

  if (warp >= C::kScoreWarp) {
  if (warp == C::kLoadWarp) {
    // ---------------------------------------------------------------- TMA producer
    int last_t[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) last_t[s] = -1;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kKVTile);
#pragma unroll
      for (int b = 0; b < D / 64; ++b) {
        tma_load_3d(sm + C::kK + b * C::kBox, &tm_k, &bars->kv_full, b * 64, j * 128, bh);
        tma_load_3d(sm + C::kV + b * C::kBox, &tm_v, &bars->kv_full, b * 64, j * 128, bh);
      }
    }
    __syncwarp();
    const bool starve = (p.flags & kBwdFlagStarveQ) != 0u;
    for (int t = 0, st = 0, ph = 0; t < n && !starve; ++t) {
      if (t >= NS && !mbar_wait_warp_inl(&bars->q_empty[st], ph ^ 1, wc)) break;
      FA_TRACE(30, t);
      if (lane == 0) {
        const int i = i0 + t;
        uint8_t* stage = sm + C::kStage0 + st * C::kStageBytes;
        float* vec = reinterpret_cast<float*>(sm + C::kVec + st * C::kVecBytes);
        mbar_arrive_expect_tx(&bars->q_full[st], 2 * C::kQTile + C::kVecBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          tma_load_3d(stage + b * C::kQBox, &tm_q, &bars->q_full[st], b * 64, i * C::kBQ, bh);
          tma_load_3d(stage + C::kQTile + b * C::kQBox, &tm_do, &bars->q_full[st], b * 64,
                      i * C::kBQ, bh);
        }
        const size_t row0 = (size_t)bh * p.T_pad + (size_t)i * C::kBQ;
        bulk_load(vec, p.lse2 + row0, C::kBQ * 4, &bars->q_full[st]);
        bulk_load(vec + C::kBQ, p.dvec + row0, C::kBQ * 4, &bars->q_full[st]);
      }
      last_t[st] = t;
      __syncwarp();
      if (++st == NS) { st = 0; ph ^= 1; }
    }
    // No copy may still be in flight when the CTA exits.
    mbar_wait_warp_inl(&bars->kv_full, 0, drain_wc);
#pragma unroll
    for (int s = 0; s < NS; ++s)
      if (last_t[s] >= 0) mbar_wait_warp_inl(&bars->q_full[s], (last_t[s] / NS) & 1, drain_wc);
  } else if (warp == C::kScoreWarp) {
    // ---------------------------------------------------------------- score issuer
    constexpr uint32_t kIdS = idesc_bf16(128, C::kBQ, false);  // Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ
    const uint32_t k_s = sbase + C::kK, v_s = sbase + C::kV;
    bool ok = mbar_wait_warp_inl(&bars->kv_full, 0, wc);
    for (int t = 0, st = 0, ph = 0; t < n && ok; ++t) {
      if (!(ok = mbar_wait_warp_inl(&bars->q_full[st], ph, wc))) break;
      if (t > 0 && !(ok = mbar_wait_warp_inl(&bars->s_free, (t - 1) & 1, wc))) break;
      FA_TRACE(1, t);
      tc_fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::kColS, kmaj(k_s, kk, C::kBox), kmaj(q_s(st), kk, C::kQBox), kIdS,
                 kk > 0);
        mma_commit(&bars->s_full);
      }
      __syncwarp();
      if (t > 0 && !(ok = mbar_wait_warp_inl(&bars->dp_free, (t - 1) & 1, wc))) break;
      FA_TRACE(2, t);
      tc_fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::kColDP, kmaj(v_s, kk, C::kBox), kmaj(do_s(st), kk, C::kQBox), kIdS,
                 kk > 0);
        mma_commit(&bars->dp_full);
        mma_commit(&bars->q_empty[st]);
      }
      __syncwarp();
      if (++st == NS) { st = 0; ph ^= 1; }
    }
    if (lane == 0) mma_commit(&bars->score_done);
    __syncwarp();
  } else if (warp == C::kGradWarp) {
    // ---------------------------------------------------------------- gradient issuer
    constexpr uint32_t kIdV = idesc_bf16(128, D, true);             // dV: A in TMEM, B MN-major
    constexpr uint32_t kIdK = idesc_bf16_ab(128, D, false, true);   // dK: A K-major, B MN-major
    // dQ (d = 64: dS·K, M = queries) or dQᵀ (d = 128: Kᵀ·dSᵀ, M = head dims): both operands
    // MN-major, N = D or kBQ.
    constexpr uint32_t kIdQ = idesc_bf16_ab(128, (D == 64) ? D : C::kBQ, true, true);
    const uint32_t k_s = sbase + C::kK;
    bool ok = true;
    for (int t = 0, st = 0; t < n && ok; ++t) {
      // dV += Pᵀ·dO_i (Pᵀ from TMEM)
      if (!(ok = mbar_wait_warp_inl(&bars->p_full, t & 1, wc))) break;
      FA_TRACE(3, t);
      tc_fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < C::kBQ / 16; ++kk)
          mma_ts(tmem + C::kColDV, tmem + C::kColP + kk * 8, mnmaj(do_s(st), kk, C::kQBox), kIdV,
                 (t > 0 || kk > 0));
        mma_commit(&bars->p_free);
      }
      __syncwarp();
      // dK += dSᵀ·Q_i, then dQ_i = dS·K_j (d = 64) or dQ_iᵀ = K_jᵀ·dSᵀ (d = 128)
      const int b = t & 1;
      const uint32_t ds_s = sbase + C::kDS + b * C::kDSBytes;
      if (!(ok = mbar_wait_warp_inl(&bars->ds_full[b], (t >> 1) & 1, wc))) break;
      if (!C::kSplitQ && t > 0 && !(ok = mbar_wait_warp_inl(&bars->dq_free, (t - 1) & 1, wc))) break;
      FA_TRACE(4, t);
      tc_fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < C::kBQ / 16; ++kk)
          mma_ss(tmem + C::kColDK, kmaj(ds_s, kk, C::kBox), mnmaj(q_s(st), kk, C::kQBox), kIdK,
                 (t > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < (C::kSplitQ ? 0 : 8); ++kk) {  // K = 128 keys
          if constexpr (D == 64)
            mma_ss(tmem + C::kColDQ, mnmaj(ds_s, kk, C::kBox), mnmaj(k_s, kk, C::kBox), kIdQ, kk > 0);
          else
            mma_ss(tmem + C::kColDQ, mnmaj(k_s, kk, C::kBox), mnmaj(ds_s, kk, C::kBox), kIdQ, kk > 0);
        }
        if constexpr (!C::kSplitQ) mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free[b]);
        mma_commit(&bars->q_empty[st]);
      }
      __syncwarp();
      if (++st == NS) st = 0;
    }
    if (lane == 0) mma_commit(&bars->grad_done);
    __syncwarp();
  } else if (C::kSplitQ && warp == C::kGradQWarp) {
    // ---------------------------------------------------------------- dQ issuer (d = 128)
    // dQ_iᵀ = K_jᵀ·dSᵀ once this tile's dSᵀ is stored and the previous dQ has been drained.
    constexpr uint32_t kIdQ = idesc_bf16_ab(128, (D == 64) ? D : C::kBQ, true, true);
    const uint32_t k_s = sbase + C::kK;
    bool ok = true;
    for (int t = 0; t < n && ok; ++t) {
      const int b = t & 1;
      const uint32_t ds_s = sbase + C::kDS + b * C::kDSBytes;
      if (!(ok = mbar_wait_warp_inl(&bars->ds_full[b], (t >> 1) & 1, wc))) break;
      if (t > 0 && !(ok = mbar_wait_warp_inl(&bars->dq_free, (t - 1) & 1, wc))) break;
      tc_fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // K = 128 keys
          if constexpr (D == 64)
            mma_ss(tmem + C::kColDQ, mnmaj(ds_s, kk, C::kBox), mnmaj(k_s, kk, C::kBox), kIdQ, kk > 0);
          else
            mma_ss(tmem + C::kColDQ, mnmaj(k_s, kk, C::kBox), mnmaj(ds_s, kk, C::kBox), kIdQ, kk > 0);
        }
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free[b]);
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(&bars->grad_done);
    __syncwarp();
  }
  teardown();
  } else if (warp >= C::kDrainWarp0) {
    // ---------------------------------------------------------------- dQ drain
    const int qd = warp & 3;
    // TMEM lane = query row (d = 64, dQ) or head dim (d = 128, dQᵀ); either way 64 columns.
    const int r = qd * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    int t = 0;
    bool ok = true;
    // 16 TMEM columns at a time through this warp's two 2 KB staging buffers, each handed to
    // the TMA engine as one bulk reduce-add (the warp's 32 lanes × 16 columns are contiguous
    // in the accumulator: 32 query rows × 16 dims at d = 64, 32 dims × 16 query rows at
    // d = 128); before a buffer is rewritten, the reduction issued from it two chunks
    // earlier must have read it.
    const uint32_t stage0 = sbase + C::kDQStage + qd * 2 * C::kDQChunk;
    int nchunk = 0;
    for (; t < n; ++t) {
      if (!(ok = mbar_wait_warp_inl(&bars->dq_full, t & 1, wc))) break;
      FA_TRACE(20, t);
      tc_fence_after_sync();
      // 32 columns at a time; the buffer is released once the last columns are in registers.
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t x[32];
        tmem_ld32(tmem + lane_off + C::kColDQ + h * 32, x);
        tmem_ld_wait();
        reg_fence32(x);
        if (h == 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->dq_free);
          FA_TRACE(21, t);
        }
        {
#pragma unroll
          for (int k2 = 0; k2 < 2; ++k2, ++nchunk) {
            const uint32_t buf = stage0 + (nchunk & 1) * C::kDQChunk;
            if (nchunk >= 2) {
              if (lane == 0) bulk_wait_group_read1();
              __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
              st_shared_v4(buf + (c * 32 + lane) * 16, x[16 * k2 + 4 * c], x[16 * k2 + 4 * c + 1],
                           x[16 * k2 + 4 * c + 2], x[16 * k2 + 4 * c + 3]);
            fence_proxy_async_smem();  // the staged values, visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
              // TMEM columns 32h + 16k2 …: column group 8h + 4k2 of lanes 32·qd …
              const int cg = 8 * h + 4 * k2;
              bulk_reduce_add_f32(p.dq_acc + ((D == 64) ? dq_acc_offset(bh, i0 + t, p.n_qt, cg, qd * 32, D)
                                                        : dq_acc_offset_t(bh, i0 + t, p.n_qt, cg, qd * 32)),
                                  buf, C::kDQChunk);
              bulk_commit_group();
            }
          }
        }
      }
    }
    if (!ok) {
      // Abandoned tiles: poison their dQ rows so that the failure cannot go unseen.
      const float nan = __int_as_float(0x7fc00000);
      for (; t < n; ++t) {
        for (int c4 = 0; c4 < 16; ++c4) {
          float* dst = p.dq_acc + ((D == 64) ? dq_acc_offset(bh, i0 + t, p.n_qt, c4, r, D)
                                             : dq_acc_offset_t(bh, i0 + t, p.n_qt, c4, r));
          red_add_v4(dst, nan, nan, nan, nan);
        }
      }
    }
    // The bulk reductions must be complete (and their sources read) before the CTA exits.
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
    teardown();
  } else {
    // ---------------------------------------------------------------- compute (warps 0-7)
    constexpr int NC = C::kNC;        // query columns of this warpgroup per tile (32)
    const int g = warp >> 2;          // columns NC·g .. NC·g + NC − 1 of each tile
    const int qd = warp & 3;
    const int r = qd * 32 + lane;     // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    // dSᵀ columns of this warpgroup: box (NC·g)/64, 16-byte chunks from ((NC·g) mod 64)/8
    const int ds_box_idx = (NC * g) / 64, ds_chunk0 = ((NC * g) % 64) / 8;
    bool ok = true;
    for (int t = 0, st = 0, ph = 0; t < n && ok; ++t) {
      const int i = i0 + t;
      const float* vec = reinterpret_cast<const float*>(sm + C::kVec + st * C::kVecBytes);
      if (!(ok = mbar_wait_warp_inl(&bars->q_full[st], ph, wc))) break;
      if (!(ok = mbar_wait_warp_inl(&bars->s_full, t & 1, wc))) break;
      FA_TRACE(10, t);
      tc_fence_after_sync();
      uint32_t s[NC];
      tmem_load_cols<NC>(tmem + lane_off + C::kColS + g * NC, s);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free);
      // Pᵀ = exp2(S·scale·log2e − log2e·LSE_q), zero where the key comes after the query
      // (the argument on fp32 pairs; the workspace holds −log2e·LSE)
      float pr[NC];
      const float4* l4 = reinterpret_cast<const float4*>(vec + g * NC);
      const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
      for (int c = 0; c < NC; c += 4) {
        const float4 l = l4[c / 4];
        float x0, x1, x2, x3;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), c2,
                         f2_pack(l.x, l.y)), x0, x1);
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), c2,
                         f2_pack(l.z, l.w)), x2, x3);
        pr[c] = ex2_approx(x0);
        pr[c + 1] = ex2_approx(x1);
        pr[c + 2] = ex2_approx(x2);
        pr[c + 3] = ex2_approx(x3);
      }
      if (CAUSAL && j * 128 + 127 > i * C::kBQ) {  // a tile the diagonal crosses
        const int rel = j * 128 + r - (i * C::kBQ + g * NC);  // key − first query of the warpgroup
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (rel > c) pr[c] = 0.f;
      }
      FA_TRACE(11, t);
      if (t >= 1 && !(ok = mbar_wait_warp_inl(&bars->p_free, (t - 1) & 1, wc))) break;
      FA_TRACE(12, t);
      uint32_t pk[NC / 2];
#pragma unroll
      for (int c = 0; c < NC / 2; ++c) pk[c] = pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
      tc_fence_after_sync();
      if constexpr (NC == 64) tmem_st32(tmem + lane_off + C::kColP + g * 32, pk);
      else if constexpr (NC == 32) tmem_st16(tmem + lane_off + C::kColP + g * 16, pk);
      else tmem_st8(tmem + lane_off + C::kColP + g * 8, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
      FA_TRACE(13, t);
      // dSᵀ = Pᵀ ∘ (dPᵀ − D_q), into shared-memory buffer t mod 2
      const int b = t & 1;
      const uint32_t ds_box = sbase + C::kDS + b * C::kDSBytes + ds_box_idx * C::kBox;
      if (!(ok = mbar_wait_warp_inl(&bars->dp_full, t & 1, wc))) break;
      FA_TRACE(14, t);
      if (t >= 2 && !(ok = mbar_wait_warp_inl(&bars->ds_free[b], ((t >> 1) - 1) & 1, wc))) break;
      FA_TRACE(15, t);
      tc_fence_after_sync();
      // dPᵀ for this warpgroup's columns (were a warpgroup to own NC = 64 columns: in two
      // halves, to stay within the register budget)
      constexpr int kDPB = (NC > 32) ? 32 : NC;  // columns per dPᵀ block
#pragma unroll
      for (int h = 0; h < NC / kDPB; ++h) {
        uint32_t dp[kDPB];
        tmem_load_cols<kDPB>(tmem + lane_off + C::kColDP + g * NC + h * kDPB, dp);
        if (h == NC / kDPB - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->dp_free);
        }
        const float4* d4 = reinterpret_cast<const float4*>(vec + C::kBQ + g * NC + h * kDPB);
#pragma unroll
        for (int q4 = 0; q4 < kDPB / 8; ++q4) {
          const float4 da = d4[2 * q4], db = d4[2 * q4 + 1];
          const int c = h * kDPB + q4 * 8;
          const uint32_t* dq8 = dp + q4 * 8;
          // dS = P ∘ (dP − D) on fp32 pairs
          const float dd[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
          float ds[8];
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            f2_unpack(f2_mul(f2_pack(pr[c + e], pr[c + e + 1]),
                             f2_sub(f2_pack(__uint_as_float(dq8[e]), __uint_as_float(dq8[e + 1])),
                                    f2_pack(dd[e], dd[e + 1]))),
                      ds[e], ds[e + 1]);
          st_row_chunk_sw128(ds_box, r, ds_chunk0 + c / 8, ds);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ds_full[b]);
      FA_TRACE(16, t);
      if (++st == NS) { st = 0; ph ^= 1; }
    }
    // ---- epilogue: warpgroup 0 writes dV_j, warpgroup 1 writes scale·dK_j (32 columns at
    // a time)
    bool done = ok && mbar_wait_warp_inl(&bars->grad_done, 0, wc) && !bars->abort;
    done = __shfl_sync(0xffffffffu, done ? 1u : 0u, 0) != 0u;  // warp-uniform (TMEM loads)
    const int key = j * 128 + r;
    tc_fence_after_sync();
    // The first half of the warpgroups writes dV, the second scale·dK, each a block of
    // D / (kCWG / 2) columns.
    constexpr int kPer = C::kCWG / 2;
    const bool is_dv = g < kPer;
    const int part = g % kPer;
    const uint32_t col = is_dv ? C::kColDV : C::kColDK;
    const float mul = is_dv ? 1.f : p.scale;
    const float nan = __int_as_float(0x7fc00000);
    __nv_bfloat16* dst = (is_dv ? p.dv : p.dk) + ((size_t)bh * p.T + key) * D;
    constexpr int kH = D / 32 / kPer;  // 32-column blocks per warpgroup
#pragma unroll
    for (int hh = 0; hh < kH; ++hh) {
      const int h = part * kH + hh;
      uint32_t x[32];
      if (done) {
        tmem_ld32(tmem + lane_off + col + h * 32, x);
        tmem_ld_wait();
      }
      reg_fence32(x);
      if (key < p.T) {
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = done ? __uint_as_float(x[c + e]) * mul : nan;
          uint4 v;
          v.x = pack_bf16x2(y[0], y[1]);
          v.y = pack_bf16x2(y[2], y[3]);
          v.z = pack_bf16x2(y[4], y[5]);
          v.w = pack_bf16x2(y[6], y[7]);
          *reinterpret_cast<uint4*>(dst + h * 32 + c) = v;
        }
      }
    }
    teardown();
  }
}

}  // namespace fa
