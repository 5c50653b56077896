// Exact attention forward for GB300 (sm_103a): tcgen05 MMAs into tensor memory, TMA
// loads through an mbarrier ring, online softmax in registers.
//
// What it computes is the exact result of softmax(scale·QKᵀ [+causal mask])·V per
// (batch, head), by the tiled scan with an online softmax described in steps ② and ③ of
// "手写 FlashAttention" (Hand-written FlashAttention, learn-llm.fim.ai ch. 19): a Q block
// stays on chip while K/V blocks stream past; per row a running max m and sum l are
// kept; when the max rises, l and the output accumulator are rescaled by
// 2^(m_old − m_new); the division by l happens once, at the end; blocks that the causal
// mask covers completely are skipped and only the diagonal block is masked element by
// element. Scores use base 2 with log2(e)·scale folded into one factor (step ④, "exp2
// and 1.4427"); the row logsumexp is emitted in natural log.
//
// One CTA = one (batch·head, pair of 128-row Q tiles). 320 threads, 10 warps:
//   warps 0-3  softmax warpgroup for Q tile 0 (thread t owns query row t, TMEM lane t)
//   warps 4-7  softmax warpgroup for Q tile 1
//   warp  8    MMA issuer (one thread) and TMEM owner
//   warp  9    TMA producer (one thread)
// Tensor memory (512 columns × 128 lanes × 32 bit):
//   [0,128)    S0 = Q0·Kᵀ (fp32), later overwritten by P0 (bf16 pairs, columns 0-63)
//   [128,256)  S1 / P1
//   [256,256+D)      O0 (fp32 accumulator)
//   [256+D,256+2D)   O1
// The two Q tiles ping-pong: while one softmax warpgroup turns its S into P, the tensor
// core computes the other tile's S or P·V.
#pragma once

#include "sm103.cuh"

namespace fa {

constexpr int kBlockM = 128;    // query rows per Q tile = TMEM lanes
constexpr int kBlockN = 128;    // keys per K/V tile
constexpr int kThreads = 320;
constexpr float kTau = 8.0f;    // lazy rescale: O and l keep a stale max until it is 2^8 too small
constexpr uint32_t kFlagStarveQ = 1u;  // FA_FLAG_TEST_STARVE_Q

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kStages = (D == 64) ? 4 : 2;      // K/V ring depth
  static constexpr int kSubBytes = kBlockM * 64 * 2;     // one 128-row × 64-col bf16 box = 16 KB
  static constexpr int kSub = D / 64;                    // boxes per tile row-block
  static constexpr int kTileBytes = kSub * kSubBytes;    // a 128×D bf16 tile
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + 1 KB alignment slack
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t never;  // stays 0: abort flag of the drain waits, which must not be cut short
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int T;
  int BH;
  int n_pairs;     // ceil(ceil(T/128)/2)
  int n_kv;        // ceil(T/128)
  float scale_log2;  // scale · log2(e)
  uint64_t timeout_ns;
  uint32_t flags;
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);

  // Heavy-first order: the first CTAs launched take the last Q-tile pairs, which under
  // the causal mask scan the most K/V tiles.
  const int L = static_cast<int>(blockIdx.x);
  const int pair = p.n_pairs - 1 - L / p.BH;
  const int bh = L % p.BH;
  const int qt0 = 2 * pair;
  int nkv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qt = qt0 + i;
    nkv[i] = (qt * kBlockM >= p.T) ? 0 : (CAUSAL ? qt + 1 : p.n_kv);
  }
  const int n_steps = max(nkv[0], nkv[1]);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->o_full[i], 1);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0u;
    bars->never = 0u;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, p.status, p.timeout_ns};

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t keep = policy_evict_last();  // K/V are re-read by this head's other Q tiles
      const bool load_q = (p.flags & kFlagStarveQ) == 0u;
      if (load_q) {
        mbar_arrive_expect_tx(&bars->q_full, 2 * C::kTileBytes);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(smem + C::kQOff + i * C::kTileBytes + s * C::kSubBytes, &tm_q,
                        &bars->q_full, s * 64, (qt0 + i) * kBlockM, bh);
      }
      int j = 0;
      for (; j < n_steps; ++j) {
        const int st = j % C::kStages;
        const int use = j / C::kStages;
        if (use > 0 && !mbar_wait(&bars->kv_empty[st], (use - 1) & 1, wc)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], C::kTileBytes);
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(smem + C::kKOff + st * C::kTileBytes + s * C::kSubBytes, &tm_k,
                           &bars->k_full[st], s * 64, j * kBlockN, bh, keep);
        mbar_arrive_expect_tx(&bars->v_full[st], C::kTileBytes);
#pragma unroll
        for (int s = 0; s < C::kSub; ++s)
          tma_load_3d_hint(smem + C::kVOff + st * C::kTileBytes + s * C::kSubBytes, &tm_v,
                           &bars->v_full[st], s * 64, j * kBlockN, bh, keep);
      }
      // Drain: every copy issued must have landed before this CTA may exit.
      const WaitCtl drain{&bars->never, nullptr, p.timeout_ns};
      if (load_q) mbar_wait(&bars->q_full, 0, drain);
      const int issued = j;
      for (int st = 0; st < C::kStages && st < issued; ++st) {
        const int last_use = (issued - 1 - st) / C::kStages;
        mbar_wait(&bars->k_full[st], last_use & 1, drain);
        mbar_wait(&bars->v_full[st], last_use & 1, drain);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false);
      constexpr uint32_t kIdescO = idesc_bf16(kBlockM, D, true);
      const uint32_t q_base = smem_u32(smem + C::kQOff);
      const uint32_t k_base = smem_u32(smem + C::kKOff);
      const uint32_t v_base = smem_u32(smem + C::kVOff);
      const uint32_t t_s[2] = {tmem + 0u, tmem + 128u};
      const uint32_t t_o[2] = {tmem + 256u, tmem + 256u + static_cast<uint32_t>(D)};

      // S_i = Q_i · K_stᵀ : M=128, N=128, K=D in steps of 16 (32 bytes inside a 128-byte
      // swizzled row; a new 16 KB box every 64 columns).
      auto issue_s = [&](int i, int st) {
        const uint32_t qa = q_base + i * C::kTileBytes;
        const uint32_t ka = k_base + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kSubBytes + (kk & 3) * 32;
          mma_ss(t_s[i], sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                 kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // O_i += P_i · V_st : A = P from TMEM (8 columns = 16 keys per step), B = V tile,
      // MN-major (D contiguous): 16 keys = 2048 bytes per step; next 64-wide column block
      // (leading byte offset) 16 KB away; next 8-key group (stride byte offset) 1 KB away.
      auto issue_pv = [&](int i, int st, bool acc) {
        const uint32_t va = v_base + st * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          mma_ts(t_o[i], t_s[i] + kk * 8, sdesc_sw128(va + kk * 2048, C::kSubBytes, 1024),
                 kIdescO, (acc || kk > 0) ? 1u : 0u);
        }
      };

      bool ok = n_steps > 0 && mbar_wait(&bars->q_full, 0, wc) && mbar_wait(&bars->k_full[0], 0, wc);
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (nkv[i] > 0) {
            issue_s(i, 0);
            mma_commit(&bars->s_full[i]);
          }
      }
      for (int j = 0; ok && j < n_steps; ++j) {
        const int st = j % C::kStages;
        if (!mbar_wait(&bars->v_full[st], (j / C::kStages) & 1, wc)) { ok = false; break; }
        const int st_next = (j + 1) % C::kStages;
        bool k_next_ready = false;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (j >= nkv[i]) continue;
          if (!mbar_wait(&bars->p_full[i], j & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
          issue_pv(i, st, j > 0);
          if (j + 1 < nkv[i]) {
            if (!k_next_ready) {
              if (!mbar_wait(&bars->k_full[st_next], ((j + 1) / C::kStages) & 1, wc)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              k_next_ready = true;
            }
            issue_s(i, st_next);
            mma_commit(&bars->s_full[i]);
          } else {
            mma_commit(&bars->o_full[i]);
          }
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[st]);
      }
      // Nothing may still be running on the tensor core when TMEM is released.
      mma_commit(&bars->mma_done);
      const WaitCtl drain{&bars->never, nullptr, p.timeout_ns};
      mbar_wait(&bars->mma_done, 0, drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qt = qt0 + wg;
    const int q_row = qt * kBlockM + row;
    const int n = nkv[wg];
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + static_cast<uint32_t>(wg * 128);
    const uint32_t t_o = tmem + lane_off + 256u + static_cast<uint32_t>(wg * D);
    const float c = p.scale_log2;

    float m_ref = -INFINITY;  // reference max (base-2 scaled units) shared by O and l
    float l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait_warp(&bars->s_full[wg], j & 1, wc)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t s[kBlockN];
#pragma unroll
      for (int c0 = 0; c0 < kBlockN; c0 += 32) tmem_ld32(t_s + c0, s + c0);
      tmem_ld_wait();
#pragma unroll
      for (int c0 = 0; c0 < kBlockN; c0 += 32) reg_fence32(s + c0);

      const int k0 = j * kBlockN;
      const bool diag = CAUSAL && (j == qt);
      if (diag || k0 + kBlockN > p.T) {
        // Keys past the end of the sequence, and (diagonal tile) keys after this query.
        const int lim = (CAUSAL ? min(q_row + 1, p.T) : p.T) - k0;
#pragma unroll
        for (int t = 0; t < kBlockN; ++t)
          if (t >= lim) s[t] = __float_as_uint(-INFINITY);
      }
      float mx0 = u2f(s[0]), mx1 = u2f(s[1]), mx2 = u2f(s[2]), mx3 = u2f(s[3]);
#pragma unroll
      for (int t = 4; t < kBlockN; t += 4) {
        mx0 = fmaxf(mx0, u2f(s[t]));
        mx1 = fmaxf(mx1, u2f(s[t + 1]));
        mx2 = fmaxf(mx2, u2f(s[t + 2]));
        mx3 = fmaxf(mx3, u2f(s[t + 3]));
      }
      const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;

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

      const float neg_m = -m_ref;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kBlockN; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float p0 = ex2_approx(fmaf(u2f(s[c0 + 2 * t]), c, neg_m));
          const float p1 = ex2_approx(fmaf(u2f(s[c0 + 2 * t + 1]), c, neg_m));
          ls0 += p0;
          ls1 += p1;
          pk[t] = pack_bf16x2(p0, p1);
        }
        tmem_st16(t_s + static_cast<uint32_t>(c0 / 2), pk);
      }
      l += ls0 + ls1;
      if (__any_sync(0xffffffffu, rescale)) {
        // Rows whose max jumped bring their accumulated O to the new reference (done
        // after P is written, when the score registers are free; O is not read by the
        // tensor core until this warp arrives on p_full below).
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(t_o + c0, r);
          tmem_ld_wait();
          reg_fence32(r);
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(u2f(r[t]) * alpha);
          tmem_st32(t_o + c0, r);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[wg]);
    }

    if (n > 0) {
      const bool good = ok && mbar_wait_warp(&bars->o_full[wg], 0, wc);
      const size_t row_idx = static_cast<size_t>(bh) * static_cast<size_t>(p.T) +
                             static_cast<size_t>(q_row);
      const bool in_range = q_row < p.T;
      uint4* orow = reinterpret_cast<uint4*>(p.o + row_idx * D);
      if (good) {
        tc_fence_after_sync();
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(t_o + c0, r);
          tmem_ld_wait();
          reg_fence32(r);
          if (in_range) {
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 16; ++t)
              pk[t] = pack_bf16x2(u2f(r[2 * t]) * inv_l, u2f(r[2 * t + 1]) * inv_l);
#pragma unroll
            for (int t = 0; t < 4; ++t)
              orow[c0 / 8 + t] = make_uint4(pk[4 * t], pk[4 * t + 1], pk[4 * t + 2], pk[4 * t + 3]);
          }
        }
        if (in_range) p.lse[row_idx] = (m_ref + log2f(l)) * 0.69314718055994530942f;
      } else if (in_range) {
        const uint32_t nan2 = 0x7FC07FC0u;  // two bf16 quiet NaNs
#pragma unroll
        for (int t = 0; t < D / 8; ++t) orow[t] = make_uint4(nan2, nan2, nan2, nan2);
        p.lse[row_idx] = __uint_as_float(0x7FC00000u);
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa
