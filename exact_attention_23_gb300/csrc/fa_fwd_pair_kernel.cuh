// Exact attention forward for GB300 (sm_103a), head dim 64, on CTA pairs: two CTAs of a
// cluster (on the two SMs of a TPC) share every tensor-core product (tcgen05 cta_group::2).
//
// It computes the same result as fa_fwd_kernel.cuh: softmax(scale·QKᵀ [+causal mask])·V per
// (batch, head) by the tiled scan with an online softmax of steps ② and ③ of "手写
// FlashAttention" (Hand-written FlashAttention, learn-llm.fim.ai ch. 19): Q tiles stay on chip
// while K/V tiles stream past, a running row max m and sum l are kept, O and l are rescaled by
// 2^(m_old − m_new) when the max rises (lazily, by more than τ), the division by l happens once
// at the end, K/V tiles the causal mask covers completely are skipped and only the diagonal
// tile is masked element by element. Scores are in base 2 with log2(e)·scale folded into one
// factor (step ④); the row logsumexp is written in natural log. The product of two CTAs, a
// low-precision-and-overlap direction of the later FlashAttention versions, is named in "内核
// 案例研究：Flash Attention" ("块稀疏注意力 V2 和 V3").
//
// Why pairs at head dim 64: a pair product computes 256 rows, each CTA supplying its own 128
// rows of A and half of B's columns. The S = Q·Kᵀ product then reads 6 KB of shared memory per
// SM and K step of 16 instead of 8 KB (74 → 65 cycles per instruction), and the N = 64 P·V
// product runs at 48 cycles instead of 61 (measured); each CTA also loads only half of every
// K and V tile.
//
// Work unit = one (batch·head, group of four 128-row Q tiles qt0…qt0+3), heaviest first,
// zig-zag over a persistent grid of pairs. Slot i ∈ {0, 1} of the pair is one 256-row product:
// the even CTA's tile qt0 + 2i and the odd CTA's tile qt0 + 2i + 1. A slot walks the K/V tiles
// its later tile needs; in the steps past its own diagonal the earlier tile's scores are all
// masked (P = 0). 352 threads per CTA, 11 warps:
//   warps 0-3  softmax of this CTA's slot-0 tile (thread t owns row t = TMEM lane t)
//   warps 4-7  softmax of this CTA's slot-1 tile
//   warp  8    S issuer of the pair (even CTA only): S_i = Q_i·Kᵀ, M = 256, N = 128; TMEM owner
//   warp  9    TMA producer: this CTA's Q tiles, its half of each K tile (64 keys) and of each
//              V tile (32 of the 64 columns)
//   warp 10    P·V issuer of the pair (even CTA only): O_i += P_i·V, M = 256, N = 64
// Tensor memory (512 columns, the same addresses in both CTAs): S_0 [0,128), S_1 [128,256),
// O_0 [256,320), O_1 [320,384), P_0 [384,448), P_1 [448,512).
// Synchronisation: the even CTA holds the barriers the issuers wait on; the odd CTA's loads
// complete on them (cta_group::2 copies) and its softmax warps arrive on them remotely. The
// issuers' commits arrive on the same barrier in both CTAs. Every wait is bounded.
#pragma once

#include "fa_fwd_kernel.cuh"

#ifndef FAP_TRACE
#define FAP_TRACE(tag, step) ((void)0)
#endif

namespace fa {

constexpr int kPairStages = 6;

struct CfgP {
  static constexpr int kQTileBytes = kBlockM * 64 * 2;   // 128 rows × 64 bf16 = 16 KB
  static constexpr int kKHalfBytes = 64 * 64 * 2;        // 64 keys × 64 bf16 = 8 KB
  static constexpr int kVHalfBytes = kBlockN * 32 * 2;   // 128 keys × 32 bf16 = 8 KB
  static constexpr int kQOff = 0;                        // 2 buffers × 2 slots
  static constexpr int kKOff = kQOff + 4 * kQTileBytes;
  static constexpr int kVOff = kKOff + kPairStages * kKHalfBytes;
  static constexpr int kOOff = kVOff + kPairStages * kVHalfBytes;  // 8 warps × 4 KB staging
  static constexpr int kPendOff = kOOff + 8 * 4096;
  static constexpr int kBarOff = kPendOff + 2 * kBlockM * 16;
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;
  static __host__ __device__ constexpr uint32_t col_s(int i) { return i ? 128u : 0u; }
  static __host__ __device__ constexpr uint32_t col_o(int i) { return 256u + (i ? 64u : 0u); }
  static __host__ __device__ constexpr uint32_t col_p(int i) { return 384u + (i ? 64u : 0u); }
};

struct BarsP {
  uint64_t q_full[2];              // even CTA: both CTAs' Q tiles of a unit landed
  uint64_t q_empty[2];             // both: the pair's S products are done with a Q buffer
  uint64_t k_full[kPairStages];    // even CTA: both halves of a K tile landed
  uint64_t v_full[kPairStages];    // even CTA: both halves of a V tile landed
  uint64_t kv_empty[kPairStages];  // both: K (S issuer) and V (P·V issuer) released
  uint64_t s_full[2];              // both: S_i computed
  uint64_t s_free[2];              // even CTA: S_i read by the 4 + 4 softmax warps
  uint64_t p_full[2];              // even CTA: P_i stored by the 4 + 4 softmax warps
  uint64_t pv_done[2];             // both: P_i·V done
  uint64_t o_free[2];              // even CTA: a unit's O_i read out by the 4 + 4 warps
  uint64_t mma_done;               // both issuers' last products done
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(BarsP) <= 512, "barrier block");

// K/V tiles a 128-row Q tile walks: all of them, or (causal) up to its diagonal; 0 past T.
__device__ __forceinline__ int steps_p(const FwdParams& p, bool causal, int qt) {
  if (qt * kBlockM >= p.T) return 0;
  return causal ? qt + 1 : p.n_kv;
}

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const FwdParams p) {
  using C = CfgP;
  constexpr int D = 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BarsP* bars = reinterpret_cast<BarsP*>(smem + C::kBarOff);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int rank = static_cast<int>(cluster_ctarank());  // 0: even CTA (issues the products)
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int n_pairs = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 8);
      mbar_init(&bars->p_full[b], 8);
      mbar_init(&bars->pv_done[b], 1);
      mbar_init(&bars->o_free[b], 8);
    }
#pragma unroll
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);
    }
    mbar_init(&bars->mma_done, 2);
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc_pair(&bars->tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  // Neither CTA's barriers may be signalled by the other before they are initialised.
  cluster_sync_all();
  tc_fence_after_sync();
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, p.status, p.timeout_ns};
  const WaitCtl drain = drain_ctl(p.timeout_ns);

  // Unit L: head bh, Q tiles qt0..qt0+3; slot i walks n[i] steps (the later tile's count).
  auto unit_at = [&](int L, int& bh, int& qt0, int& n0, int& n1) {
    const int pos = static_cast<int>(p.div_bh.div(static_cast<uint32_t>(L)));
    bh = L - pos * p.BH;
    qt0 = (p.n_units - 1 - pos) * 4;
    n0 = max(steps_p(p, CAUSAL, qt0), steps_p(p, CAUSAL, qt0 + 1));
    n1 = max(steps_p(p, CAUSAL, qt0 + 2), steps_p(p, CAUSAL, qt0 + 3));
  };

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
    }
    const uint64_t keep = policy_evict_last();
    int g = 0, qn = 0;
    bool ok = true;
    for (int r = 0; ok && r * n_pairs < p.total_units; ++r) {
      const int L = unit_index(r, pair, n_pairs);
      if (L >= p.total_units) continue;
      int bh, qt0, n0, n1;
      unit_at(L, bh, qt0, n0, n1);
      const int qb = qn & 1;
      if (qn >= 2 && !mbar_wait_warp(&bars->q_empty[qb], ((qn >> 1) - 1) & 1, wc)) { ok = false; break; }
      if (leader) {
        uint8_t* qdst = smem + C::kQOff + qb * 2 * C::kQTileBytes;
        if (rank == 0) {
          mbar_arrive_expect_tx(&bars->q_full[qb], 4 * C::kQTileBytes);  // both CTAs' tiles
#pragma unroll
          for (int i = 0; i < 2; ++i)
            tma_load_3d(qdst + i * C::kQTileBytes, &tm_q, &bars->q_full[qb], 0, (qt0 + 2 * i) * kBlockM, bh);
        } else {
          const uint32_t qf = mapa_shared(&bars->q_full[qb], 0);
#pragma unroll
          for (int i = 0; i < 2; ++i)
            tma_load_3d_pair(qdst + i * C::kQTileBytes, &tm_q, qf, 0, (qt0 + 2 * i + 1) * kBlockM, bh, keep);
        }
      }
      __syncwarp();
      ++qn;
      const int n = max(n0, n1);
      for (int j = 0; j < n; ++j, ++g) {
        const int st = g % kPairStages;
        const int use = g / kPairStages;
        if (use > 0 && !mbar_wait_warp(&bars->kv_empty[st], (use - 1) & 1, wc)) { ok = false; break; }
        if (leader) {
          uint8_t* kdst = smem + C::kKOff + st * C::kKHalfBytes;
          uint8_t* vdst = smem + C::kVOff + st * C::kVHalfBytes;
          // this CTA's 64 of the tile's 128 keys, and its 32 of the 64 value columns
          if (rank == 0) {
            mbar_arrive_expect_tx(&bars->k_full[st], 2 * C::kKHalfBytes);
            tma_load_3d_hint(kdst, &tm_k, &bars->k_full[st], 0, j * kBlockN, bh, keep);
            mbar_arrive_expect_tx(&bars->v_full[st], 2 * C::kVHalfBytes);
            tma_load_3d_hint(vdst, &tm_v, &bars->v_full[st], 0, j * kBlockN, bh, keep);
          } else {
            tma_load_3d_pair(kdst, &tm_k, mapa_shared(&bars->k_full[st], 0), 0, j * kBlockN + 64, bh, keep);
            tma_load_3d_pair(vdst, &tm_v, mapa_shared(&bars->v_full[st], 0), 32, j * kBlockN, bh, keep);
          }
        }
        __syncwarp();
      }
    }
    // The even CTA's drain waits for the last use of every barrier, which counts both CTAs'
    // bytes; the closing cluster barrier then keeps the odd CTA alive until they landed.
    if (rank == 0) {
      for (int b = 0; b < 2 && b < qn; ++b) mbar_wait_warp(&bars->q_full[b], ((qn - 1 - b) >> 1) & 1, drain);
      for (int st = 0; st < kPairStages && st < g; ++st) {
        const int last_use = (g - 1 - st) / kPairStages;
        mbar_wait_warp(&bars->k_full[st], last_use & 1, drain);
        mbar_wait_warp(&bars->v_full[st], last_use & 1, drain);
      }
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    if (rank == 0) {
      const bool leader = lane == 0;
      auto commit = [&](uint64_t* bar) {
        if (leader) mma_commit_pair(bar);
        __syncwarp();
      };
      bool ok = true;
      if (warp == 8) {
        const uint32_t idesc = idesc_bf16(2 * kBlockM, kBlockN, false) | p.s_negate;
        const uint32_t q_base = smem_u32(smem + C::kQOff);
        const uint32_t k_base = smem_u32(smem + C::kKOff);
        int g = 0, qn = 0;
        int ns[2] = {0, 0};
        for (int r = 0; ok && r * n_pairs < p.total_units; ++r) {
          const int L = unit_index(r, pair, n_pairs);
          if (L >= p.total_units) continue;
          int bh, qt0, n0, n1;
          unit_at(L, bh, qt0, n0, n1);
          const int qb = qn & 1;
          if (!mbar_wait_warp(&bars->q_full[qb], (qn >> 1) & 1, wc)) { ok = false; break; }
          const int n = max(n0, n1);
          for (int j = 0; j < n; ++j, ++g) {
            const int st = g % kPairStages;
            if (!mbar_wait_warp(&bars->k_full[st], (g / kPairStages) & 1, wc)) { ok = false; break; }
            tc_fence_after_sync();
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (j >= (i ? n1 : n0)) continue;
              // S_i may be overwritten once both CTAs' softmax warps have read it.
              if (ns[i] > 0) {
                if (!mbar_wait_warp(&bars->s_free[i], (ns[i] - 1) & 1, wc)) { ok = false; break; }
                tc_fence_after_sync();
              }
              if (leader) {
                const uint32_t qa = q_base + (qb * 2 + i) * C::kQTileBytes;
                const uint32_t ka = k_base + st * C::kKHalfBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                  mma_ss_pair(tmem + C::col_s(i), sdesc_sw128(qa + kk * 32, 16, 1024),
                              sdesc_sw128(ka + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
                mma_commit_pair(&bars->s_full[i]);
              }
              __syncwarp();
              ++ns[i];
            }
            if (!ok) break;
            commit(&bars->kv_empty[st]);  // K(j) is free once these products are done
          }
          if (!ok) break;
          commit(&bars->q_empty[qb]);
          ++qn;
        }
      } else {
        // B = V half, MN-major: 32 columns (64 bytes, one 64-byte swizzle atom) per key row,
        // 8-key groups 512 bytes apart, 16 keys = 1 KB per instruction.
        const uint32_t idesc = idesc_bf16(2 * kBlockM, D, true);
        const uint32_t v_base = smem_u32(smem + C::kVOff);
        int g = 0;
        int np[2] = {0, 0}, nunits[2] = {0, 0};
        for (int r = 0; ok && r * n_pairs < p.total_units; ++r) {
          const int L = unit_index(r, pair, n_pairs);
          if (L >= p.total_units) continue;
          int bh, qt0, n0, n1;
          unit_at(L, bh, qt0, n0, n1);
          const int n = max(n0, n1);
          int jt[2] = {0, 0};
          for (int j = 0; j < n; ++j, ++g) {
            const int st = g % kPairStages;
            if (!mbar_wait_warp(&bars->v_full[st], (g / kPairStages) & 1, wc)) { ok = false; break; }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (j >= (i ? n1 : n0)) continue;
              if (jt[i] == 0 && nunits[i] > 0) {
                if (!mbar_wait_warp(&bars->o_free[i], (nunits[i] - 1) & 1, wc)) { ok = false; break; }
              }
              if (!mbar_wait_warp(&bars->p_full[i], np[i] & 1, wc)) { ok = false; break; }
              tc_fence_after_sync();
              if (leader) {
                const uint32_t va = v_base + st * C::kVHalfBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk)
                  mma_ts_pair(tmem + C::col_o(i), tmem + C::col_p(i) + kk * 8,
                              sdesc_sw64(va + kk * 1024, 8192, 512), idesc,
                              (jt[i] > 0 || kk > 0) ? 1u : 0u);
                mma_commit_pair(&bars->pv_done[i]);
              }
              __syncwarp();
              ++np[i];
              ++jt[i];
            }
            if (!ok) break;
            commit(&bars->kv_empty[st]);  // V(j) is free once these products are done
          }
#pragma unroll
          for (int i = 0; i < 2; ++i)
            if ((i ? n1 : n0) > 0) ++nunits[i];
        }
      }
      commit(&bars->mma_done);
      mbar_wait_warp(&bars->mma_done, 0, drain);
    }
  } else {
    // ------------------------------------------------------------ softmax (both CTAs)
    const int wg = warp >> 2;  // slot
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::col_s(wg);
    const uint32_t t_o = tmem + lane_off + C::col_o(wg);
    const uint32_t t_p = tmem + lane_off + C::col_p(wg);
    const float c = p.scale_log2;
    // Arrivals on the even CTA's barriers: local there, remote from the odd CTA.
    const uint32_t s_free_rem = mapa_shared(&bars->s_free[wg], 0);
    const uint32_t p_full_rem = mapa_shared(&bars->p_full[wg], 0);
    const uint32_t o_free_rem = mapa_shared(&bars->o_free[wg], 0);
    auto arrive_even = [&](uint64_t* local, uint32_t remote) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(local);
        else mbar_arrive_remote_relaxed(remote);
      }
    };

    int gs = 0;  // S_wg consumed so far over the pair's units
    bool ok = true;
    struct RowOut {
      size_t row_idx;
      int r0, bh;
      bool in_range;
    };
    auto fail_rows = [&](const RowOut& w) {
      if (!w.in_range) return;
      uint4* orow = reinterpret_cast<uint4*>(p.o + w.row_idx * D);
      const uint32_t nan2 = 0x7FC07FC0u;
#pragma unroll
      for (int t = 0; t < D / 8; ++t) orow[t] = make_uint4(nan2, nan2, nan2, nan2);
      p.lse[w.row_idx] = __uint_as_float(0x7FC00000u);
    };
    // A finished unit's O (its last P·V done) to the output through this warp's staging slice
    // and a TMA store (rows past T not written); O is released to the next unit's first P·V
    // as soon as it has been read.
    auto epilogue = [&](const RowOut& w, float l, float m) {
      uint32_t o[D];
      tmem_ld32(t_o, o);
      tmem_ld32(t_o + 32, o + 32);
      tmem_ld_wait();
      reg_fence32(o);
      reg_fence32(o + 32);
      arrive_even(&bars->o_free[wg], o_free_rem);
      const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
      uint8_t* slice = smem + C::kOOff + (wg * 4 + quad) * 4096;
      const uint32_t ob = smem_u32(slice) + lane * 128;
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        st_shared_v4(ob + ((ch ^ (lane & 7)) << 4),
                     pack_bf16x2(u2f(o[8 * ch]) * inv_l, u2f(o[8 * ch + 1]) * inv_l),
                     pack_bf16x2(u2f(o[8 * ch + 2]) * inv_l, u2f(o[8 * ch + 3]) * inv_l),
                     pack_bf16x2(u2f(o[8 * ch + 4]) * inv_l, u2f(o[8 * ch + 5]) * inv_l),
                     pack_bf16x2(u2f(o[8 * ch + 6]) * inv_l, u2f(o[8 * ch + 7]) * inv_l));
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && w.r0 < p.T) {
        tma_store_3d(&tm_o, slice, 0, w.r0, w.bh);
        bulk_commit_group();
      }
      if (w.in_range) p.lse[w.row_idx] = (m + log2f(l)) * 0.69314718055994530942f;
    };
    bool pend = false;
    float4* const prec = reinterpret_cast<float4*>(smem + C::kPendOff) + wg * kBlockM + row;
    auto parked = [&](float& l, float& m) {
      const float4 v = *prec;
      l = v.x;
      m = v.y;
      const int r0 = __float_as_int(v.z), bh = __float_as_int(v.w);
      const int q_row = r0 + lane;
      return RowOut{static_cast<size_t>(bh) * static_cast<size_t>(p.T) + static_cast<size_t>(q_row),
                    r0, bh, q_row < p.T};
    };
    auto fail_pending = [&]() {
      float l, m;
      fail_rows(parked(l, m));
      pend = false;
    };
    // The pending unit's last P·V was step gs − 1 of this slot.
    auto flush_pending = [&]() -> bool {
      if (!mbar_wait_warp(&bars->pv_done[wg], (gs - 1) & 1, wc)) return false;
      tc_fence_after_sync();
      float l, m;
      const RowOut w = parked(l, m);
      epilogue(w, l, m);
      pend = false;
      return true;
    };

    for (int r = 0; r * n_pairs < p.total_units; ++r) {
      const int L = unit_index(r, pair, n_pairs);
      if (L >= p.total_units) continue;
      int bh, qt0, n0, n1;
      unit_at(L, bh, qt0, n0, n1);
      const int n = wg ? n1 : n0;
      if (n == 0) continue;
      const int qt = qt0 + 2 * wg + rank;       // this CTA's tile in the slot
      const int n_own = steps_p(p, CAUSAL, qt);  // steps holding keys its rows may see
      const int q_row = qt * kBlockM + row;
      const RowOut cur{static_cast<size_t>(bh) * static_cast<size_t>(p.T) + static_cast<size_t>(q_row),
                       qt * kBlockM + quad * 32, bh, q_row < p.T};
      if (!ok) {
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      float m_ref = -INFINITY;
      float l = 0.0f;
      for (int j = 0; j < n; ++j, ++gs) {
        if (!mbar_wait_warp(&bars->s_full[wg], gs & 1, wc)) { ok = false; break; }
        FAP_TRACE(30 + wg, j);
        tc_fence_after_sync();
        const int k0 = j * kBlockN;
        // Keys past T, (causal) keys after this query, and every key of a step past this
        // tile's own diagonal (its slot partner needs it; these rows see none of it).
        const int lim = (j >= n_own) ? 0 : (CAUSAL ? min(q_row + 1, p.T) : p.T) - k0;
        const bool masked = (j >= n_own) || (CAUSAL && j == qt) || (k0 + kBlockN > p.T);
        uint32_t s[kBlockN];
        tmem_ld32(t_s + 0, s);
        tmem_ld32(t_s + 32, s + 32);
        tmem_ld32(t_s + 64, s + 64);
        tmem_ld32(t_s + 96, s + 96);
        tmem_ld_wait();
        reg_fence32(s);
        reg_fence32(s + 32);
        reg_fence32(s + 64);
        reg_fence32(s + 96);
        arrive_even(&bars->s_free[wg], s_free_rem);
        if (masked) {
#pragma unroll
          for (int t = 0; t < kBlockN; ++t)
            if (t >= lim) s[t] = __float_as_uint(-INFINITY);
        }
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = fmaxf(u2f(s[2 * a]), u2f(s[2 * a + 1]));
#pragma unroll
        for (int t = 16; t < kBlockN; t += 16)
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
        const uint64_t c2 = f2_pack(c, c);
        // (rows of a tile past T see no key at all: m_ref = −∞, their p are 0)
        const float m_use = (m_ref == -INFINITY) ? 0.0f : m_ref;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int t = 0; t < kBlockN / 2; ++t) {
          const uint64_t x2 = f2_fma(f2_pack(u2f(s[2 * t]), u2f(s[2 * t + 1])), c2, nm2);
          float x0, x1;
          f2_unpack(x2, x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          if (t & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
          else acc0 = f2_add(acc0, f2_pack(p0, p1));
          pk[t] = pack_bf16x2(p0, p1);
        }
        bool waited = false;
        if (any_rescale) {
          // Rows whose max jumped bring O to the new reference before this step's P·V (rare);
          // O must hold every earlier step (the previous P·V done; j ≥ 1, so this unit's).
          if (!mbar_wait_warp(&bars->pv_done[wg], (gs - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
          waited = true;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 16) {
            uint32_t o[16];
            tmem_ld16(t_o + c0, o);
            tmem_ld_wait();
            reg_fence16(o);
#pragma unroll
            for (int t = 0; t < 16; ++t) o[t] = __float_as_uint(u2f(o[t]) * alpha);
            tmem_st16(t_o + c0, o);
          }
        }
        // P_wg's columns are free once the previous P·V has read them.
        if (gs > 0 && !waited) {
          if (!mbar_wait_warp(&bars->pv_done[wg], (gs - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
        }
        tmem_st32(t_p, pk);
        tmem_st32(t_p + 32, pk + 32);
        tmem_st_wait();
        arrive_even(&bars->p_full[wg], p_full_rem);
        FAP_TRACE(22 + wg, j);
        {
          float a0, a1, b0, b1;
          f2_unpack(acc0, a0, a1);
          f2_unpack(acc1, b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        // (j = 0) the previous unit's last P·V was the one waited for above: write it out.
        if (j == 0 && pend) {
          tc_fence_after_sync();
          float pl, pm;
          const RowOut w = parked(pl, pm);
          epilogue(w, pl, pm);
          pend = false;
        }
      }
      if (!ok) {
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      *prec = make_float4(l, m_ref, __int_as_float(cur.r0), __int_as_float(cur.bh));
      pend = true;
    }
    if (pend) {
      if (!(ok && flush_pending())) fail_pending();
    }
    if (lane == 0) bulk_wait_group_read0();
  }

  tc_fence_before_sync();
  __syncthreads();
  // Both CTAs stay until every product and every copy of the pair is done.
  cluster_sync_all();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace fa
