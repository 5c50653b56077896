// Exact attention forward for GB300 (sm_103a), one 128-row Q tile per CTA with the score
// and probability tiles double-buffered in tensor memory.
//
// It computes the same result as fa_fwd_kernel.cuh, softmax(scale·QKᵀ [+causal mask])·V per
// (batch, head) by the tiled scan with an online softmax of steps ② and ③ of "手写
// FlashAttention" (Hand-written FlashAttention, learn-llm.fim.ai ch. 19): the Q tile stays on
// chip while K/V tiles stream past, a running row max m and sum l are kept, O and l are
// rescaled by 2^(m_old − m_new) when the max rises (lazily, by more than τ), the division by l
// happens once at the end, blocks the causal mask covers completely are skipped and only the
// diagonal block is masked element by element. Scores are in base 2 with log2(e)·scale folded
// into one factor (step ④); the row logsumexp is written in natural log.
//
// Why one tile with two buffers: with one S and one P region per tile, every K step of a tile
// is a chain of hand-offs between warps (S read → next S issued → done → read; P stored →
// P·V issued → done → next P stored), and two such tiles ping-ponging on one SM left the
// softmax warps waiting on those hand-offs for most of each step. Here S(j+1) is computed into
// the other S region while the softmax works on S(j), and P(j) is stored into the P region
// P·V(j−1) is not reading, so the softmax warps find their next S ready and their P region
// free, and the tensor core always has the next product queued.
//
// Work unit = one (batch·head, 128-row Q tile), heaviest first, zig-zag over a persistent grid
// (one CTA per SM). The general form (GEN: queries against a longer key sequence with
// bottom-right causal visibility, a key range per unit, a block mask) walks, per unit, only
// the K tiles of its range that its rows use, and writes the range's normalised fp32 row and
// LSE when the key range is split (merged afterwards by fa_fwd_combine_kernel).
//
// Softmax halves (H = 2 at D = 64, H = 1 at D = 128). At D = 64 each query row's 128 keys of
// a step are split over two warps that own the same TMEM lanes: warp q (q = 0…3) takes keys
// 0–63 and warp q + 4 keys 64–127 of every K tile, and each half keeps its own running max,
// sum and O accumulator over its keys — the tiled scan of step ③ of the same page applied to
// two interleaved key subsets — so the two warps never meet inside the step loop. They merge
// once per unit (O = (2^(m₀−m)·O₀ + 2^(m₁−m)·O₁) / (2^(m₀−m)·l₀ + 2^(m₁−m)·l₁), m = max(m₀, m₁)),
// exchanging m and l through shared memory. Two softmax warps per SM sub-partition hide each
// other's latency, where one warp with a whole 128-key row sat in its own dependency chains.
// Warps (32·(4H + 3) threads):
//   warps 0 … 4H−1  softmax: warp w owns query rows 32(w mod 4) … +31 (TMEM lanes) and the
//                   keys 64·(w div 4) … of each step when H = 2
//   warp  4H        S issuer: S(j) = Q·K(j)ᵀ into S[j mod 2] (one elected thread); TMEM owner
//   warp  4H + 1    TMA producer (Q per unit; K and V per step through a ring)
//   warp  4H + 2    P·V issuer: O_h += P_h(j)·V_h(j) from P[j mod 2]
// With 224 threads (H = 1) every thread may hold 255 registers, with 352 (H = 2) 168: either
// way the softmax keeps its part of the S row, its P and its state in registers without
// spilling.
// Tensor memory (512 columns × 128 lanes × 32 bit):
//   [0,128) S[0]   [128,256) S[1]   [256,256+H·D) O_0 … O_{H−1} (fp32)   then P[0], P[1] (64
//   columns each: 128 keys as bf16 pairs, half h in columns 32h … of each) — 512 columns.
// Every barrier phase is counted over the CTA's whole list of units, so units follow one
// another with no re-initialisation; a unit's epilogue (O / l to bf16 through shared memory
// and a TMA store, and the LSE) is deferred into the first step of the next unit.
#pragma once

#include "fa_fwd_kernel.cuh"

// Timeline hooks: compiled out unless a tracing build defines FA1_TRACE(tag, step).
#ifndef FA1_TRACE
#define FA1_TRACE(tag, step) ((void)0)
#endif

namespace fa {

template <int D>
struct Cfg1 {
  static_assert(D == 64 || D == 128, "head dim");
  // Softmax halves: two O accumulators fit tensor memory at D = 64 only.
  static constexpr int kHalves = (D == 64) ? 2 : 1;
  static constexpr int kCols = kBlockN / kHalves;        // keys per softmax warp and step
  static constexpr int kSoftWarps = 4 * kHalves;
  static constexpr int kWarpS = kSoftWarps;              // S issuer, TMEM owner
  static constexpr int kWarpLoad = kSoftWarps + 1;       // TMA producer
  static constexpr int kWarpPV = kSoftWarps + 2;         // P·V issuer
  static constexpr int kThreads = (kSoftWarps + 3) * 32;
  // K/V ring depth: four stages at D = 64; D = 128 tiles are twice the size, two fit.
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static_assert(kStages >= 2 && kStages <= 4, "K/V ring depth (barrier arrays hold 4)");
  static constexpr int kQBufs = 2;                       // this unit's Q and the next one's
  static constexpr int kSubBytes = kBlockM * 64 * 2;     // one 128-row × 64-col bf16 box = 16 KB
  static constexpr int kSub = D / 64;
  static constexpr int kTileBytes = kSub * kSubBytes;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBufs * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  // Output staging: each softmax warp's 32 rows × 64 columns (one 4 KB box of the O tensor
  // map, 128-byte swizzle); D = 128 goes out in two rounds.
  static constexpr int kOOff = kVOff + kStages * kTileBytes;
  static constexpr int kOBytes = 4 * 4096;
  // Each softmax thread's deferred epilogue record (l, m, first row of its warp, head).
  static constexpr int kPendOff = kOOff + kOBytes;
  // The halves' (m, l) exchange at the end of a unit, double-buffered by unit parity.
  static constexpr int kXchOff = kPendOff + kHalves * kBlockM * 16;
  static constexpr int kBarOff = kXchOff + 2 * kHalves * kBlockM * 8;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + 1 KB alignment slack
  static __host__ __device__ constexpr uint32_t col_s(int b) { return b ? 128u : 0u; }
  static __host__ __device__ constexpr uint32_t col_o(int h) { return 256u + h * D; }
  static __host__ __device__ constexpr uint32_t col_p(int b) {
    return 256u + kHalves * D + (b ? 64u : 0u);
  }
  static_assert(256 + kHalves * D + 128 <= 512, "tensor memory columns");
};

struct Bars1 {
  uint64_t q_full[2];    // a unit's Q tile landed (producer -> S issuer)
  uint64_t q_empty[2];   // the S issuer is done with a Q buffer (tensor core -> producer)
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4];  // two arrivals per use: K released by the S issuer, V by the P·V issuer
  uint64_t s_full[2];    // S(j) computed into S[j mod 2] (tensor core -> softmax)
  uint64_t s_free[2];    // S[b] read into registers (4 softmax warps -> S issuer)
  uint64_t p_full[2];    // P(j) stored into P[j mod 2], O rescaled if needed (softmax -> P·V)
  uint64_t pv_done[2];   // P·V(j) done: P[j mod 2] reusable, O holds steps ≤ j (tensor core)
  uint64_t o_free;       // a unit's O has been read out (softmax -> P·V issuer)
  uint64_t mma_done;
  uint64_t xch[4][2];    // halves: both warps of lanes 32q… posted (m, l) (unit parity)
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(Bars1) <= 512, "barrier block");

template <int D, bool CAUSAL, bool GEN = false>
__global__ void __launch_bounds__(Cfg1<D>::kThreads, 1)
    fa_fwd1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdParams p) {
  using C = Cfg1<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars1* bars = reinterpret_cast<Bars1*>(smem + C::kBarOff);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int cta = static_cast<int>(blockIdx.x);
  const int grid = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], C::kSoftWarps);
      mbar_init(&bars->p_full[b], C::kSoftWarps);
      mbar_init(&bars->pv_done[b], 1);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);
    }
    mbar_init(&bars->o_free, C::kSoftWarps);
    mbar_init(&bars->mma_done, 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      mbar_init(&bars->xch[q][0], 2);
      mbar_init(&bars->xch[q][1], 2);
    }
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == C::kWarpS) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // Launched as a programmatic dependent: the set-up above overlapped the previous kernel's
  // tail; nothing in global memory is touched before that kernel has completed.
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, p.status, p.timeout_ns};
  const WaitCtl drain = drain_ctl(p.timeout_ns);

  if (warp == C::kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
    }
    const uint64_t keep = policy_evict_last();  // K/V are re-read by this head's other Q tiles
    const bool load_q = (p.flags & kFlagStarveQ) == 0u;
    const bool later_q = (p.flags & kFlagStarveLaterQ) == 0u;
    int g = 0, qn = 0, ql = 0;
    bool ok = true;
    for (int r = 0; ok && r * grid < p.total_units; ++r) {
      const int L = unit_index(r, cta, grid);
      if (L >= p.total_units) continue;
      const Unit u = unit_of<CAUSAL, GEN>(p, L);
      const int qb = qn & 1;
      if (qn >= 2 && !mbar_wait_warp(&bars->q_empty[qb], ((qn >> 1) - 1) & 1, wc)) { ok = false; break; }
      const bool load = load_q && (later_q || qn == 0);
      if (load) ++ql;
      if (load && leader) {
        mbar_arrive_expect_tx(&bars->q_full[qb], C::kTileBytes);
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d(smem + C::kQOff + qb * C::kTileBytes + s * C::kSubBytes, &tm_q,
                      &bars->q_full[qb], s * 64, u.qt0 * kBlockM, u.bh);
      }
      __syncwarp();
      ++qn;
      UnitSteps<CAUSAL, GEN> us;
      us.begin(p, u);
      for (int j = 0; j < u.n_steps; ++j, ++g) {
        us.next(u, j);
        const int kt = us.kt;
        const int st = g % C::kStages;
        const int use = g / C::kStages;
        if (use > 0 && !mbar_wait_warp(&bars->kv_empty[st], (use - 1) & 1, wc)) { ok = false; break; }
        if (leader) {
          mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
#pragma unroll
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d_hint(smem + C::kKOff + st * C::kTileBytes + s * C::kSubBytes, &tm_k,
                             &bars->k_full[st], s * 64, kt * kBlockN, u.bh, keep);
          mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
#pragma unroll
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d_hint(smem + C::kVOff + st * C::kTileBytes + s * C::kSubBytes, &tm_v,
                             &bars->v_full[st], s * 64, kt * kBlockN, u.bh, keep);
        }
        __syncwarp();
      }
    }
    // Drain: every copy issued must have landed before this CTA may exit.
    for (int b = 0; b < 2 && b < ql; ++b) {
      const int last = (ql - 1 - b) >> 1;  // last loaded use of Q buffer b
      mbar_wait_warp(&bars->q_full[b], last & 1, drain);
    }
    for (int st = 0; st < C::kStages && st < g; ++st) {
      const int last_use = (g - 1 - st) / C::kStages;
      mbar_wait_warp(&bars->k_full[st], last_use & 1, drain);
      mbar_wait_warp(&bars->v_full[st], last_use & 1, drain);
    }
  } else if (warp == C::kWarpS || warp == C::kWarpPV) {
    // ------------------------------------------------------------ MMA issuers
    const bool leader = lane == 0;
    auto commit = [&](uint64_t* bar) {
      if (leader) mma_commit(bar);
      __syncwarp();
    };
    bool ok = true;
    if (warp == C::kWarpS) {
      // S(j) = Q·K(j)ᵀ : M=128, N=128, K=D in steps of 16 (32 bytes inside a 128-byte
      // swizzled row; a new 16 KB box every 64 columns), into S[j mod 2].
      const uint32_t idesc = idesc_bf16(kBlockM, kBlockN, false) | p.s_negate;
      const uint32_t q_base = smem_u32(smem + C::kQOff);
      const uint32_t k_base = smem_u32(smem + C::kKOff);
      int g = 0, qn = 0;
      for (int r = 0; ok && r * grid < p.total_units; ++r) {
        const int L = unit_index(r, cta, grid);
        if (L >= p.total_units) continue;
        const Unit u = unit_of<CAUSAL, GEN>(p, L);
        const int qb = qn & 1;
        if (!mbar_wait_warp(&bars->q_full[qb], (qn >> 1) & 1, wc)) { ok = false; break; }
        for (int j = 0; j < u.n_steps; ++j, ++g) {
          const int st = g % C::kStages;
          const int b = g & 1;
          if (!mbar_wait_warp(&bars->k_full[st], (g / C::kStages) & 1, wc)) { ok = false; break; }
          // S[b] may be overwritten once the softmax has read S(g − 2) out of it.
          FA1_TRACE(3, j);
          if (g >= 2 && !mbar_wait_warp(&bars->s_free[b], ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          FA1_TRACE(5, j);
          tc_fence_after_sync();
          if (leader) {
            const uint32_t qa = q_base + qb * C::kTileBytes;
            const uint32_t ka = k_base + st * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::kSubBytes + (kk & 3) * 32;
              mma_ss(tmem + C::col_s(b), sdesc_sw128(qa + off, 16, 1024),
                     sdesc_sw128(ka + off, 16, 1024), idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[b]);
            mma_commit(&bars->kv_empty[st]);  // K(j) is free once this product is done
          }
          __syncwarp();
          FA1_TRACE(16, j);
        }
        if (!ok) break;
        commit(&bars->q_empty[qb]);  // this unit's Q is free once its S products are done
        ++qn;
      }
    } else {
      // O_h += P_h(j)·V_h(j) : A = P from TMEM (8 columns = 16 keys per step), B = V tile,
      // MN-major (D contiguous): 16 keys = 2048 bytes per step; next 64-wide column block
      // (leading byte offset) 16 KB away; next 8-key group (stride byte offset) 1 KB away.
      // Half h takes the keys 64h … of the tile into its own accumulator.
      const uint32_t idesc = idesc_bf16(kBlockM, D, true);
      const uint32_t v_base = smem_u32(smem + C::kVOff);
      int g = 0, nunits = 0;
      for (int r = 0; ok && r * grid < p.total_units; ++r) {
        const int L = unit_index(r, cta, grid);
        if (L >= p.total_units) continue;
        const Unit u = unit_of<CAUSAL, GEN>(p, L);
        for (int j = 0; j < u.n_steps; ++j, ++g) {
          const int st = g % C::kStages;
          const int b = g & 1;
          if (!mbar_wait_warp(&bars->v_full[st], (g / C::kStages) & 1, wc)) { ok = false; break; }
          FA1_TRACE(8, j);
          if (!mbar_wait_warp(&bars->p_full[b], (g >> 1) & 1, wc)) { ok = false; break; }
          FA1_TRACE(11, j);
          // A unit's first P·V overwrites O: the previous unit's O must have been read out.
          if (j == 0 && nunits > 0 && !mbar_wait_warp(&bars->o_free, (nunits - 1) & 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (leader) {
            const uint32_t va = v_base + st * C::kTileBytes;
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
              for (int kk = 0; kk < C::kCols / 16; ++kk)
                mma_ts(tmem + C::col_o(h), tmem + C::col_p(b) + h * (C::kCols / 2) + kk * 8,
                       sdesc_sw128(va + (h * (C::kCols / 16) + kk) * 2048, C::kSubBytes, 1024),
                       idesc, (j > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars->pv_done[b]);
            mma_commit(&bars->kv_empty[st]);  // V(j) is free once this product is done
          }
          __syncwarp();
          FA1_TRACE(14, j);
        }
        if (u.n_steps > 0) ++nunits;  // (a general-form unit may use no K tile: no P·V)
      }
    }
    // Nothing may still be running on the tensor core when TMEM is released.
    commit(&bars->mma_done);
    mbar_wait_warp(&bars->mma_done, 0, drain);
  } else if (warp < C::kSoftWarps) {
    // ------------------------------------------------------------ softmax warps
    constexpr int H = C::kHalves;
    constexpr int kC = C::kCols;              // keys of a step this warp owns
    const int quad = warp & 3;                // TMEM lanes 32·quad … (query rows)
    const int half = warp >> 2;               // keys kC·half … of each step (H = 2)
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_o = tmem + lane_off + C::col_o(half);
    const float c = p.scale_log2;

    int g = 0;    // K steps consumed so far over this CTA's units
    int ne = 0;   // epilogues done (unit parity of the halves' exchange)
    bool ok = true;
    // Where a unit's rows go: the bf16 output (row_idx; r0 = the warp's first row, for the
    // TMA store) and LSE, or (general form with several key ranges) the fp32 partial row
    // and LSE of its range (part_idx). With two halves each warp writes half of the columns.
    struct RowOut {
      size_t row_idx, part_idx;
      int r0, bh;
      bool in_range, partial;
    };
    auto row_out = [&](int bh, int split, int r0) {
      const int q_row = r0 + lane;
      return RowOut{static_cast<size_t>(bh) * static_cast<size_t>(p.T) + static_cast<size_t>(q_row),
                    (static_cast<size_t>(split) * p.BH + bh) * static_cast<size_t>(p.T) +
                        static_cast<size_t>(q_row),
                    r0, bh, q_row < p.T, GEN && p.n_splits > 1};
    };
    constexpr int kOutCols = D / H;           // output columns this warp writes
    const int c_out = half * kOutCols;
    auto write_lse = [&](const RowOut& w, float v) {
      if (!w.in_range || half != 0) return;
      if (w.partial) p.lse_part[w.part_idx] = v;
      else p.lse[w.row_idx] = v;
    };
    // A row that saw no key (general form: O = 0, LSE = −∞) or a failed unit (NaN).
    auto write_const_row = [&](const RowOut& w, uint32_t bits) {
      if (!w.in_range) return;
      if (w.partial) {
        float4* prow = reinterpret_cast<float4*>(p.o_part + w.part_idx * D + c_out);
        const float f = u2f(bits);
#pragma unroll
        for (int t = 0; t < kOutCols / 4; ++t) prow[t] = make_float4(f, f, f, f);
      } else {
        uint4* orow = reinterpret_cast<uint4*>(p.o + w.row_idx * D + c_out);
        const uint32_t b2 = pack_bf16x2(u2f(bits), u2f(bits));
#pragma unroll
        for (int t = 0; t < kOutCols / 8; ++t) orow[t] = make_uint4(b2, b2, b2, b2);
      }
    };
    auto fail_rows = [&](const RowOut& w) {
      write_const_row(w, 0x7FC00000u);
      write_lse(w, __uint_as_float(0x7FC00000u));
    };
    // The finished unit's O (TMEM, after its last P·V) to the output; O is released to the
    // next unit's first P·V as soon as it has been read. (General form: a row that saw no
    // key of the range has l = 0 and gets O = 0, LSE = −∞; partial rows go out as fp32, each
    // thread writing its own row.)
    //
    // H = 1: read 32 columns at a time, scale by 1/l, stage in this warp's 4 KB slice in the
    // O map's 128-byte-swizzled layout (16-byte chunk c of row r at c ^ (r mod 8)), one TMA
    // store per 64 columns; rows past the sequence are not written.
    //
    // H = 2: the two warps of a row post their (m, l) in shared memory and meet on an
    // mbarrier (bounded wait); each then reads its 32 output columns of both accumulators,
    // merges them with the weights 2^(m_h − m) / l and writes them straight to memory.
    // Returns false when the meeting gave up (the rows are then written as failed).
    auto epilogue = [&](const RowOut& w, float l, float m) -> bool {
      if constexpr (H == 2) {
        const int par = ne & 1;
        float2* xs = reinterpret_cast<float2*>(smem + C::kXchOff) + (par * H) * kBlockM;
        xs[half * kBlockM + row] = make_float2(m, l);
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->xch[quad][par]);
        const bool met = mbar_wait_warp(&bars->xch[quad][par], (ne >> 1) & 1, wc);
        ++ne;
        if (!met) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->o_free);
          fail_rows(w);
          return false;
        }
        const float2 other = xs[(1 - half) * kBlockM + row];
        const float m0 = half ? other.x : m, l0 = half ? other.y : l;
        const float m1 = half ? m : other.x, l1 = half ? l : other.y;
        const float M = fmaxf(m0, m1);
        const float f0 = (m0 == -INFINITY) ? 0.0f : ex2_approx(m0 - M);
        const float f1 = (m1 == -INFINITY) ? 0.0f : ex2_approx(m1 - M);
        const float L = l0 * f0 + l1 * f1;
        const float inv_l = (GEN && !(L > 0.0f)) ? 0.0f : 1.0f / L;
        const float w0 = f0 * inv_l, w1 = f1 * inv_l;
        uint32_t o0[32], o1[32];
        tmem_ld32(tmem + lane_off + C::col_o(0) + c_out, o0);
        tmem_ld32(tmem + lane_off + C::col_o(1) + c_out, o1);
        tmem_ld_wait();
        reg_fence32(o0);
        reg_fence32(o1);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free);
        if (w.in_range) {
          if (w.partial) {
            float4* prow = reinterpret_cast<float4*>(p.o_part + w.part_idx * D + c_out);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              prow[t] = make_float4(fmaf(u2f(o0[4 * t]), w0, u2f(o1[4 * t]) * w1),
                                    fmaf(u2f(o0[4 * t + 1]), w0, u2f(o1[4 * t + 1]) * w1),
                                    fmaf(u2f(o0[4 * t + 2]), w0, u2f(o1[4 * t + 2]) * w1),
                                    fmaf(u2f(o0[4 * t + 3]), w0, u2f(o1[4 * t + 3]) * w1));
          } else {
            uint4* orow = reinterpret_cast<uint4*>(p.o + w.row_idx * D + c_out);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              uint32_t pk4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = 8 * t + 2 * e;
                pk4[e] = pack_bf16x2(fmaf(u2f(o0[x]), w0, u2f(o1[x]) * w1),
                                     fmaf(u2f(o0[x + 1]), w0, u2f(o1[x + 1]) * w1));
              }
              orow[t] = make_uint4(pk4[0], pk4[1], pk4[2], pk4[3]);
            }
          }
        }
        write_lse(w, (GEN && !(L > 0.0f)) ? -INFINITY : (M + log2f(L)) * 0.69314718055994530942f);
        return true;
      } else {
        const float inv_l = (GEN && !(l > 0.0f)) ? 0.0f : 1.0f / l;
        uint8_t* slice = smem + C::kOOff + warp * 4096;
        const uint32_t ob = smem_u32(slice) + lane * 128;
#pragma unroll 1
        for (int hb = 0; hb < D / 64; ++hb) {
          uint32_t o[64];
          tmem_ld32(t_o + hb * 64, o);
          tmem_ld32(t_o + hb * 64 + 32, o + 32);
          tmem_ld_wait();
          reg_fence32(o);
          reg_fence32(o + 32);
          if (hb == D / 64 - 1) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->o_free);
          }
          if (GEN && w.partial) {
            if (w.in_range) {
              float4* prow = reinterpret_cast<float4*>(p.o_part + w.part_idx * D + hb * 64);
#pragma unroll
              for (int t = 0; t < 16; ++t)
                prow[t] = make_float4(u2f(o[4 * t]) * inv_l, u2f(o[4 * t + 1]) * inv_l,
                                      u2f(o[4 * t + 2]) * inv_l, u2f(o[4 * t + 3]) * inv_l);
            }
            continue;
          }
          if (lane == 0) bulk_wait_group_read0();  // the slice's previous store has read it
          __syncwarp();
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(ob + ((ch ^ (lane & 7)) << 4),
                         pack_bf16x2(u2f(o[8 * ch]) * inv_l, u2f(o[8 * ch + 1]) * inv_l),
                         pack_bf16x2(u2f(o[8 * ch + 2]) * inv_l, u2f(o[8 * ch + 3]) * inv_l),
                         pack_bf16x2(u2f(o[8 * ch + 4]) * inv_l, u2f(o[8 * ch + 5]) * inv_l),
                         pack_bf16x2(u2f(o[8 * ch + 6]) * inv_l, u2f(o[8 * ch + 7]) * inv_l));
          fence_proxy_async_smem();  // the staged rows, visible to the TMA engine
          __syncwarp();
          if (lane == 0 && w.r0 < p.T) {
            tma_store_3d(&tm_o, slice, hb * 64, w.r0, w.bh);
            bulk_commit_group();
          }
        }
        write_lse(w, (GEN && !(l > 0.0f)) ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f);
        return true;
      }
    };
    // The pending (finished, not yet written) unit's l, m and output position wait in this
    // thread's 16-byte record in shared memory, not in registers the step loop needs.
    bool pend = false;
    float4* const prec = reinterpret_cast<float4*>(smem + C::kPendOff) + half * kBlockM + row;
    // (.w = bh + BH·split)
    auto parked = [&](float& l, float& m) {
      const float4 v = *prec;
      l = v.x;
      m = v.y;
      const int r0 = __float_as_int(v.z), hs = __float_as_int(v.w);
      const int split = GEN ? hs / p.BH : 0;
      return row_out(hs - split * p.BH, split, r0);
    };
    auto fail_pending = [&]() {
      float l, m;
      fail_rows(parked(l, m));
      pend = false;
    };
    // Finishes the pending unit once its last P·V (step g − 1) is done.
    auto flush_pending = [&]() {
      if (ok && mbar_wait_warp(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc)) {
        tc_fence_after_sync();
        float l, m;
        const RowOut w = parked(l, m);
        if (!epilogue(w, l, m)) ok = false;
        pend = false;
      } else {
        ok = false;
        fail_pending();
      }
    };

    for (int r = 0; r * grid < p.total_units; ++r) {
      const int L = unit_index(r, cta, grid);
      if (L >= p.total_units) continue;
      const Unit u = unit_of<CAUSAL, GEN>(p, L);
      const int n = u.nkv[0];
      const int qt = u.qt0;
      const int q_row = qt * kBlockM + row;
      const RowOut cur = row_out(u.bh, u.split, qt * kBlockM + quad * 32);
      if (!ok) {
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      if (GEN && n == 0) {  // the unit uses no K tile of its range
        if (pend) flush_pending();
        write_const_row(cur, 0u);
        write_lse(cur, -INFINITY);
        continue;
      }
      float m_ref = -INFINITY;  // reference max (base-2 scaled units) shared by O_h and l
      float l = 0.0f;
      // the tile's K tiles (GEN: its walk, the next position fetched a step ahead)
      Walk w{nullptr, 0};
      int nx = 0;
      if constexpr (GEN) {
        w = walk_of<CAUSAL>(p, u, 0);
        nx = walk_next(w, u.kb - 1);
      }
      int kt = u.kb - 1;  // (dense: u.kb = 0, step j is K tile j)
      for (int j = 0; j < n; ++j, ++g) {
        if constexpr (GEN) {
          kt = nx;
          nx = walk_next(w, kt);
        } else {
          ++kt;
        }
        const int b = g & 1;
        if (!mbar_wait_warp(&bars->s_full[b], (g >> 1) & 1, wc)) { ok = false; break; }
        FA1_TRACE(30, j);
        tc_fence_after_sync();
        const int k0 = kt * kBlockN + half * kC;
        // Keys past the end of the sequence, and (causal) keys after this query (general
        // form: after query + Tk − Tq).
        int lim;
        bool masked;
        if constexpr (GEN) {
          lim = (CAUSAL ? min(q_row + 1 + p.kv_off, p.Tk) : p.Tk) - k0;
          masked = lim < kC;
        } else {
          lim = (CAUSAL ? min(q_row + 1, p.T) : p.T) - k0;
          masked = (CAUSAL && kt == qt) || (k0 + kC > p.T);
        }
        uint32_t s[kC];
        const uint32_t t_s = tmem + lane_off + C::col_s(b) + half * kC;
#pragma unroll
        for (int c0 = 0; c0 < kC; c0 += 32) tmem_ld32(t_s + c0, s + c0);
        tmem_ld_wait();
#pragma unroll
        for (int c0 = 0; c0 < kC; c0 += 32) reg_fence32(s + c0);
        // S(g) is in registers: the tensor core may compute S(g + 2) into this region.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[b]);
        FA1_TRACE(20, j);
        if (masked) {
#pragma unroll
          for (int t = 0; t < kC; ++t)
            if (t >= lim) s[t] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = fmaxf(u2f(s[2 * a]), u2f(s[2 * a + 1]));
#pragma unroll
        for (int t = 16; t < kC; t += 16)
#pragma unroll
          for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], u2f(s[t + 2 * a]), u2f(s[t + 2 * a + 1]));
        const float m_tile =
            fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * c;

        float alpha = 1.0f;
        bool rescale = false;
        if (j == 0) {
          m_ref = m_tile;
        } else if (m_tile > m_ref + kTau) {
          alpha = ex2_approx(m_ref - m_tile);
          m_ref = m_tile;
          l *= alpha;
          rescale = true;
        }
        const bool any_rescale = __any_sync(0xffffffffu, rescale);
        FA1_TRACE(40, j);

        // p = 2^(s·c − m_ref) on fp32 pairs; row sum in fp32; P kept as bf16 pairs. (A row
        // whose keys so far are all masked — the general form, or a half at the causal
        // diagonal — has m_ref = −∞ and all its p are 0.)
        const uint64_t c2 = f2_pack(c, c);
        const float m_use = ((GEN || H == 2) && m_ref == -INFINITY) ? 0.0f : m_ref;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
        uint32_t pk[kC / 2];
#pragma unroll
        for (int t = 0; t < kC / 2; ++t) {
          const uint64_t x2 = f2_fma(f2_pack(u2f(s[2 * t]), u2f(s[2 * t + 1])), c2, nm2);
          float x0, x1;
          f2_unpack(x2, x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          if (t & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
          else acc0 = f2_add(acc0, f2_pack(p0, p1));
          pk[t] = pack_bf16x2(p0, p1);
        }
        FA1_TRACE(42, j);
        if (any_rescale) {
          // Rows whose max jumped bring their O_h to the new reference before this step's
          // P·V (rare: the reference moves only by more than τ). O_h must hold every earlier
          // step: the previous P·V done (j ≥ 1, so it belongs to this unit).
          if (!mbar_wait_warp(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tmem_ld32(t_o + c0, o);
            tmem_ld_wait();
            reg_fence32(o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(u2f(o[t]) * alpha);
            tmem_st32(t_o + c0, o);
          }
        }
        // P[b] is free once P·V(g − 2) has read it.
        if (g >= 2) {
          if (!mbar_wait_warp(&bars->pv_done[b], ((g >> 1) - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
        }
        FA1_TRACE(44, j);
        const uint32_t t_p = tmem + lane_off + C::col_p(b) + half * (kC / 2);
#pragma unroll
        for (int c0 = 0; c0 < kC / 2; c0 += 32) tmem_st32(t_p + c0, pk + c0);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[b]);
        FA1_TRACE(22, j);
        {
          float a0, a1, b0, b1;
          f2_unpack(acc0, a0, a1);
          f2_unpack(acc1, b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        // (j = 0) The previous unit's last P·V, step g − 1, is the one before this step's:
        // read its O out (releasing O to this unit's first P·V) and write it.
        if (j == 0 && pend) {
          // The previous unit ended at step g − 1.
          if (mbar_wait_warp(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, wc)) {
            tc_fence_after_sync();
            float pl, pm;
            const RowOut w = parked(pl, pm);
            pend = false;
            if (!epilogue(w, pl, pm)) {
              ok = false;
              break;
            }
          } else {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      *prec = make_float4(l, m_ref, __int_as_float(cur.r0), __int_as_float(cur.bh + p.BH * u.split));
      pend = true;
    }
    if (pend) flush_pending();  // the last unit's epilogue (its last step is g − 1)
    // The output rows' TMA stores must have read their shared-memory source before the
    // CTA exits (their global writes complete with the grid).
    if (lane == 0) bulk_wait_group_read0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::kWarpS) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
