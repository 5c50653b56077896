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
// Work unit = one (batch·head, pair of 128-row Q tiles). The kernel is persistent: one
// CTA per SM walks a strided list of units, so that the next unit's Q/K/V loads and first
// S = Q·Kᵀ overlap the current unit's epilogue, and TMEM/barrier set-up happens once.
// 352 threads, 11 warps:
//   warps 0-3  softmax warpgroup for Q tile 0 (thread t owns query row t, TMEM lane t)
//   warps 4-7  softmax warpgroup for Q tile 1
//   warp  8    S issuer: S_i = Q_i·Kᵀ MMAs (one elected thread); TMEM owner
//   warp  9    TMA producer
//   warp 10    P·V issuer: O_i += P_i·V MMAs (one elected thread)
// The two issuers run independently so that neither's barrier waits leave the tensor
// core idle: a tcgen05.mma batch that starts on an idle tensor pipe pays several hundred
// cycles of start-up, so the pipe is kept fed from two queues.
// Tensor memory (512 columns × 128 lanes × 32 bit):
//   [0,128)          S0 = Q0·Kᵀ (fp32)
//   [128,256)        S1
//   [256,256+D)      O0 (fp32 accumulator)
//   [256+D,256+2D)   O1
//   D = 64:  [384,448) P0, [448,512) P1 (bf16 pairs). Because P has its own columns, the
//            next S = Q·Kᵀ is issued as soon as the softmax has read the current S into
//            registers, and runs on the tensor core while that softmax is still working.
//   D = 128: no room: P_i overwrites the first 64 columns of S_i, so the next S_i waits
//            until P_i·V has consumed P_i.
// Every barrier phase is counted over the CTA's whole list of units (each role walks the
// same list and keeps the same running counts), so units follow one another with no
// re-initialisation.
// A unit's output leaves through shared memory: each softmax warp stages its 32 rows in
// the O tensor map's swizzled layout and issues a TMA store. At D = 64 the epilogue is
// deferred into the tile's first step of the next unit, after that step's P store, so that
// the tensor core does not wait on it; at D = 128, P is stored and P·V issued in two
// halves of the keys. (Both are described where they happen.)
#pragma once

#include "sm103.cuh"

// Timeline hooks: compiled out unless a tracing build defines FA_TRACE(tag, step).
#ifndef FA_TRACE
#define FA_TRACE(tag, step) ((void)0)
#endif

namespace fa {

constexpr int kBlockM = 128;    // query rows per Q tile = TMEM lanes
constexpr int kBlockN = 128;    // keys per K/V tile
constexpr int kThreads = 352;
constexpr float kTau = 8.0f;    // lazy rescale: O and l keep a stale max until it is 2^8 too small
constexpr uint32_t kFlagStarveQ = 1u;       // FA_FLAG_TEST_STARVE_Q
constexpr uint32_t kFlagStarveLaterQ = 2u;  // FA_FLAG_TEST_STARVE_LATER_Q

template <int D, bool QK8 = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  // K/V ring depth (measured: 3 beats 2, 4 and 6 at d=64; d = 128 in bf16 has room for 2;
  // with e4m3 Q/K tiles half the size, 3)
  static constexpr int kStages = (D == 64 || QK8) ? 3 : 2;
  static_assert(kStages >= 1 && kStages <= 4, "K/V ring depth (barrier arrays hold 4)");
  static constexpr int kQBufs = (D == 64) ? 2 : 1;       // Q tile pairs in flight (next unit's Q)
  static constexpr int kSubBytes = kBlockM * 64 * 2;     // one 128-row × 64-col bf16 box = 16 KB
  static constexpr int kSub = D / 64;                    // boxes per tile row-block
  static constexpr int kTileBytes = kSub * kSubBytes;    // a 128×D bf16 tile
  // Q and K tiles: bf16 as above, or (QK8) one box of 128 rows × D one-byte e4m3 codes,
  // swizzled in 128-byte (D = 128) or 64-byte (D = 64) rows.
  static constexpr int kQKSub = QK8 ? 1 : kSub;
  static constexpr int kQKSubBytes = QK8 ? kBlockM * D : kSubBytes;
  static constexpr int kQKTileBytes = kQKSub * kQKSubBytes;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBufs * 2 * kQKTileBytes;
  static constexpr int kVOff = kKOff + kStages * kQKTileBytes;
  // Output staging: each softmax warp's 32 rows × 64 columns (4 KB, one box of the O tensor
  // map, 128-byte swizzle) go through shared memory to one TMA store; D = 128 takes two
  // rounds. (Written row by row from registers, every warp store touched 32 rows, and an
  // epilogue's stores held the warp's next barrier poll back by about a thousand cycles.)
  static constexpr int kOOff = kVOff + kStages * kTileBytes;
  static constexpr int kOBytes = 8 * 4096;
  // D = 64: each softmax thread's deferred epilogue (l, m, first row of its warp, head).
  static constexpr bool kDefer = (D == 64);
  static constexpr int kPendOff = kOOff + kOBytes;
  static constexpr int kBarOff = kPendOff + (kDefer ? 2 * kBlockM * 16 : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // barriers + 1 KB alignment slack
  // P is stored, and P·V issued, in kPParts parts of the keys. D = 128: two halves, so the
  // first half's P·V (four N = 128 products) runs while the second is exponentiated
  // (measured +6 %; four quarters measured 15 % slower than halves). D = 64: one part
  // (halves measured 15 % slower: the extra wait and commit between two short batches of
  // N = 64 products cost more than they hide).
  static constexpr int kPParts = (D == 128) ? 2 : 1;
  static_assert(kPParts == 1 || kPParts == 2 || kPParts == 4, "P parts (barrier arrays hold 4)");
  // Tensor-memory columns (see the layout at the top of this file).
  static constexpr bool kSepP = (D == 64);
  static __device__ __forceinline__ constexpr uint32_t col_s(int i) { return i ? 128u : 0u; }
  static __device__ __forceinline__ constexpr uint32_t col_o(int i) { return 256u + (i ? D : 0u); }
  static __device__ __forceinline__ constexpr uint32_t col_p(int i) {
    return kSepP ? (i ? 448u : 384u) : col_s(i);
  }
};

struct Bars {
  uint64_t q_full[2];   // a unit's Q tiles landed (producer -> S issuer)
  uint64_t q_empty[2];  // the S issuer is done with a Q buffer (tensor core -> producer)
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t kv_empty[4]; // two arrivals per use: K released by the S issuer, V by the P·V issuer
  uint64_t s_full[2];   // S_i computed (tensor core -> softmax)
  uint64_t s_free[2];   // S_i read into registers (softmax -> S issuer); D = 64 only
  uint64_t p_full[2][4];   // [i][h]: part h of P_i's keys stored, O_i rescaled if needed
                          // (softmax -> P·V issuer)
  uint64_t pv_part[2][3];  // [i][h]: parts 0..h of P_i·V done: their keys of P_i reusable
  uint64_t pv_done[2];  // P_i·V done: P_i reusable, O_i stable (tensor core -> softmax)
  uint64_t o_free[2];   // a unit's O_i has been read out (softmax -> P·V issuer)
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Division of 32-bit unsigned numerators by a fixed divisor d ≥ 1 without a divide: with
// m = ⌈2⁶⁴ / d⌉, ⌊n / d⌋ = ⌊m·n / 2⁶⁴⌋ for every n < 2³² (Lemire, Kaser and Kurz, "Faster
// remainder by direct computation", 2019, theorem 1). d = 1 is taken apart (m would not fit).
struct FastDiv {
  uint64_t m;
  uint32_t d;
  static FastDiv make(uint32_t d) { return FastDiv{d > 1u ? ~0ull / d + 1ull : 0ull, d}; }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    return d == 1u ? n : static_cast<uint32_t>(__umul64hi(m, n));
#else
    return d == 1u ? n : static_cast<uint32_t>((static_cast<unsigned __int128>(m) * n) >> 64);
#endif
  }
};

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  int* status;
  int T;
  int BH;
  int n_units;        // Q-tile groups per (batch, head): ceil(n_kv / tiles_per_cta)
  int total_units;    // n_units · BH
  int n_kv;           // ceil(T/128): K/V tiles, also Q tiles
  int tiles_per_cta;  // 2 (ping-pong pair) or 1 (short sequences: more CTAs)
  FastDiv div_bh;     // division by BH
  FastDiv div_splits; // division by n_splits (general form)
  float scale_log2;   // |scale| · log2(e) (the smallest normal float when scale = 0)
  uint32_t s_negate;  // kIdescNegateA when scale < 0 (S = −Q·Kᵀ, so that S·scale_log2 keeps its
                      // sign), else 0
  uint64_t timeout_ns;
  uint32_t flags;
  // General form only (GEN kernels; T above is then the query length Tq):
  int Tk;             // key length
  int n_qt;           // ceil(Tq/128) query tiles
  int kv_off;         // Tk − Tq: causal visibility is key ≤ query + kv_off (bottom-right)
  int n_splits;       // key ranges per query unit (partial results when > 1)
  int kt_per_split;   // K tiles per range
  const uint8_t* bmask;  // optional [mask heads][n_qt][n_kv] block mask (nonzero = keep)
  int bmask_heads;    // 1 (shared) or BH
  float* o_part;      // n_splits > 1: [n_splits][BH][Tq][D] fp32 normalised partial O
  float* lse_part;    // n_splits > 1: [n_splits][BH][Tq] fp32 partial LSE (−∞: no key)
};

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// One work unit. Units are numbered heaviest first (under the causal mask the cost of a
// Q-tile pair grows with its position), all heads at one position together. CTA c takes
// the units of round r = 0, 1, 2, ... at position c in even rounds
// and G−1−c in odd rounds (G = grid size). Over a list sorted by cost this zig-zag gives
// every CTA nearly the same total work without any shared counter.
//
// General form (GEN): a unit is (head, query unit, key range). Its steps walk the K tiles
// of the range that at least one of its Q tiles uses; tile i uses K tile kt when the tile
// exists, kt is not past the last key its rows may see (causal, bottom-right), and the
// block mask keeps (qt, kt). nkv[i] counts those steps for tile i, n_steps the union.
struct Unit {
  int bh, qt0, nkv[2], n_steps;
  int kb, ke;     // K-tile range [kb, ke) (dense: [0, n_steps))
  int last[2];    // last K tile visible to tile i (GEN, causal)
  int split, mh;  // key-range index; block-mask head
};

__device__ __forceinline__ int unit_index(int round, int cta, int grid) {
  return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// General form: the K tiles of a unit's range that Q tile i uses, walked by a cursor over
// the tile's block-mask row. The cursor keeps two values (the row, the end of the tile's
// visible keys) instead of the unit, and callers fetch the next position a step ahead of
// its use, so the mask byte's load is not on the step's critical path.
struct Walk {
  const uint8_t* mrow;  // block-mask row of the tile (nullptr: every K tile)
  int end;              // past the last K tile the tile may use (range end, causal limit)
};
constexpr int kNoTile = 0x7fffffff;

template <bool CAUSAL>
__device__ __forceinline__ Walk walk_of(const FwdParams& p, const Unit& u, int i) {
  // (ternaries, not u.last[i]: a runtime index would move the unit to local memory)
  const int qt = u.qt0 + i;
  const bool exists = i < p.tiles_per_cta && qt * kBlockM < p.T;
  const int last = i ? u.last[1] : u.last[0];
  Walk w;
  w.end = !exists ? u.kb : (CAUSAL ? min(u.ke, last + 1) : u.ke);
  w.mrow = p.bmask ? p.bmask + (static_cast<size_t>(u.mh) * p.n_qt + qt) * p.n_kv : nullptr;
  return w;
}

// The first K tile after kt that the walk uses, kNoTile when none is left.
__device__ __forceinline__ int walk_next(const Walk& w, int kt) {
  for (++kt; kt < w.end; ++kt)
    if (w.mrow == nullptr || w.mrow[kt] != 0) return kt;
  return kNoTile;
}

template <bool CAUSAL, bool GEN>
__device__ __forceinline__ Unit unit_of(const FwdParams& p, int L) {
  Unit u;
  if constexpr (GEN) {
    // bh fastest, then key range, then query unit, the last query unit first (under the
    // causal mask later query tiles see more keys: the heaviest units go out first)
    const int rest = static_cast<int>(p.div_bh.div(static_cast<uint32_t>(L)));
    u.bh = L - rest * p.BH;
    const int qu = static_cast<int>(p.div_splits.div(static_cast<uint32_t>(rest)));
    u.split = rest - qu * p.n_splits;
    u.qt0 = (p.n_units - 1 - qu) * p.tiles_per_cta;
    u.kb = u.split * p.kt_per_split;
    u.ke = min(p.n_kv, u.kb + p.kt_per_split);
    u.mh = (p.bmask_heads == 1) ? 0 : u.bh;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int last_row = min((u.qt0 + i) * kBlockM + kBlockM - 1, p.T - 1);
      u.last[i] = CAUSAL ? min(p.n_kv - 1, (last_row + p.kv_off) / kBlockN) : p.n_kv - 1;
    }
    const Walk w0 = walk_of<CAUSAL>(p, u, 0), w1 = walk_of<CAUSAL>(p, u, 1);
    if (p.bmask == nullptr) {  // every K tile of [kb, end_i): contiguous
      u.nkv[0] = max(0, w0.end - u.kb);
      u.nkv[1] = max(0, w1.end - u.kb);
      u.n_steps = max(u.nkv[0], u.nkv[1]);
    } else {
      u.nkv[0] = u.nkv[1] = u.n_steps = 0;
      const int hi = max(w0.end, w1.end);
      for (int kt = u.kb; kt < hi; ++kt) {
        const bool a0 = kt < w0.end && w0.mrow[kt] != 0;
        const bool a1 = kt < w1.end && w1.mrow[kt] != 0;
        u.nkv[0] += a0;
        u.nkv[1] += a1;
        u.n_steps += (a0 || a1);
      }
    }
    return u;
  }
  u.kb = 0;
  u.split = 0;
  u.mh = 0;
  const int pos = static_cast<int>(p.div_bh.div(static_cast<uint32_t>(L)));
  u.bh = L - pos * p.BH;
  const int idx = p.n_units - 1 - pos;
  u.qt0 = idx * p.tiles_per_cta;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qt = u.qt0 + i;
    u.nkv[i] = (i >= p.tiles_per_cta || qt * kBlockM >= p.T) ? 0 : (CAUSAL ? qt + 1 : p.n_kv);
  }
  u.n_steps = max(u.nkv[0], u.nkv[1]);
  u.ke = u.n_steps;
  u.last[0] = u.last[1] = 0;
  return u;
}

// General form: the steps of a unit for a role that follows both tiles (producer, MMA
// issuers). Step j is K tile kt, the smaller of the two tiles' next K tiles, and tile i takes
// part when act[i]. (Dense units need none of this: step j is K tile j, and tile i is active
// while j < nkv[i].)
template <bool CAUSAL, bool GEN>
struct UnitSteps {
  Walk w[2];
  int nx[2];
  int kt;
  bool act[2];
  __device__ __forceinline__ void begin(const FwdParams& p, const Unit& u) {
    kt = -1;
    if constexpr (GEN) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        w[i] = walk_of<CAUSAL>(p, u, i);
        nx[i] = walk_next(w[i], u.kb - 1);
      }
    }
  }
  __device__ __forceinline__ void next(const Unit& u, int j) {
    if constexpr (GEN) {
      kt = min(nx[0], nx[1]);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        act[i] = nx[i] == kt;
        if (act[i]) nx[i] = walk_next(w[i], kt);  // (the next position, a step ahead)
      }
    } else {
      kt = j;
      act[0] = j < u.nkv[0];
      act[1] = j < u.nkv[1];
    }
  }
};

// QK8: Q and K arrive as e4m3 codes (their per-tensor scales folded into scale_log2) and
// S = Q·Kᵀ runs as a kind::f8f6f4 product; V, P and O are as in the bf16 path.
template <int D, bool CAUSAL, bool GEN = false, bool QK8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using C = Cfg<D, QK8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOff);

  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int cta = static_cast<int>(blockIdx.x);
  const int grid = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->q_full[b], 1);
      mbar_init(&bars->q_empty[b], 1);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 2);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
#pragma unroll
      for (int h = 0; h < 4; ++h) mbar_init(&bars->p_full[i][h], 4);
#pragma unroll
      for (int h = 0; h < 3; ++h) mbar_init(&bars->pv_part[i][h], 1);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->o_free[i], 4);
    }
    mbar_init(&bars->mma_done, 2);
    bars->abort = 0u;
    fence_mbar_init();
  }
  if (warp == 8) {
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
  // Bounded warp waits. At d = 64 (bf16) lane 0 alone polls: a waiting control warp then
  // takes fewer issue slots from the softmax warps on its sub-partition (0.9 % faster); the
  // e4m3 kernel, whose waits sit closer to its critical path, keeps every lane polling.
  auto wait_w = [](uint64_t* bar, uint32_t parity, const WaitCtl& w) {
    if constexpr (D == 64 && !QK8) return mbar_wait_warp_lp(bar, parity, w);
    else return mbar_wait_warp(bar, parity, w);
  };

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (uniform control flow); lane 0 issues the copies.
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
    int g = 0;       // K/V steps issued so far (over this CTA's units)
    int qn = 0;      // Q tile pairs issued so far
    int ql = 0;      // ... of which loaded (fewer only under the test flags)
    bool ok = true;
    for (int r = 0; ok && r * grid < p.total_units; ++r) {
      const int L = unit_index(r, cta, grid);
      if (L >= p.total_units) continue;
      const Unit u = unit_of<CAUSAL, GEN>(p, L);
      const int qb = qn % C::kQBufs;
      if (qn >= C::kQBufs &&
          !wait_w(&bars->q_empty[qb], ((qn / C::kQBufs) - 1) & 1, wc)) { ok = false; break; }
      const bool load = load_q && (later_q || qn == 0);
      if (load) ++ql;
      if (load && leader) {
        mbar_arrive_expect_tx(&bars->q_full[qb], p.tiles_per_cta * C::kQKTileBytes);
        for (int i = 0; i < p.tiles_per_cta; ++i)
#pragma unroll
          for (int s = 0; s < C::kQKSub; ++s)
            tma_load_3d(smem + C::kQOff + (qb * 2 + i) * C::kQKTileBytes + s * C::kQKSubBytes, &tm_q,
                        &bars->q_full[qb], s * 64, (u.qt0 + i) * kBlockM, u.bh);
      }
      __syncwarp();
      ++qn;
      UnitSteps<CAUSAL, GEN> us;
      if constexpr (GEN) us.begin(p, u);
      int kt = u.kb - 1;
      for (int j = 0; j < u.n_steps; ++j, ++g) {
        if constexpr (GEN) {
          us.next(u, j);
          kt = us.kt;
        } else {
          ++kt;
        }
        const int st = g % C::kStages;
        const int use = g / C::kStages;
        if (use > 0 && !wait_w(&bars->kv_empty[st], (use - 1) & 1, wc)) { ok = false; break; }
        FA_TRACE(1, j);
        if (leader) {
          mbar_arrive_expect_tx(&bars->k_full[st], C::kQKTileBytes);
#pragma unroll
          for (int s = 0; s < C::kQKSub; ++s)
            tma_load_3d_hint(smem + C::kKOff + st * C::kQKTileBytes + s * C::kQKSubBytes, &tm_k,
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
    // (Q was loaded for the CTA's first ql units; buffer b served every kQBufs-th of them.)
    for (int b = 0; b < C::kQBufs && b < ql; ++b) {
      const int last = (ql - 1 - b) / C::kQBufs;  // last loaded use of buffer b
      wait_w(&bars->q_full[b], last & 1, drain);
    }
    for (int st = 0; st < C::kStages && st < g; ++st) {
      const int last_use = (g - 1 - st) / C::kStages;
      wait_w(&bars->k_full[st], last_use & 1, drain);
      wait_w(&bars->v_full[st], last_use & 1, drain);
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // The whole warp runs the schedule and waits (uniform control flow); lane 0 alone
    // issues each batch of tcgen05.mma and the commit that tracks it.
    const bool leader = lane == 0;
    auto commit = [&](uint64_t* bar) {
      if (leader) mma_commit(bar);
      __syncwarp();
    };
    if (warp == 8) {
      // S_i = Q_i · K_stᵀ : M=128, N=128, K=D in steps of 16 (32 bytes inside a 128-byte
      // swizzled row; a new 16 KB box every 64 columns). Committed to s_full[i].
      const uint32_t kIdescS = idesc_bf16(kBlockM, kBlockN, false) | p.s_negate;
      const uint32_t q_base = smem_u32(smem + C::kQOff);
      const uint32_t k_base = smem_u32(smem + C::kKOff);
      auto issue_s = [&](int qb, int i, int st) {
        if (leader) {
          const uint32_t qa = q_base + (qb * 2 + i) * C::kQKTileBytes;
          const uint32_t ka = k_base + st * C::kQKTileBytes;
          if constexpr (QK8) {
            // e4m3: K = 32 codes = 32 bytes per instruction inside one swizzled row
            const uint32_t kIdescS8 = idesc_e4m3(kBlockM, kBlockN) | p.s_negate;
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
              const uint32_t off = kk * 32;
              const uint64_t da = (D == 128) ? sdesc_sw128(qa + off, 16, 1024) : sdesc_sw64(qa + off, 16, 512);
              const uint64_t db = (D == 128) ? sdesc_sw128(ka + off, 16, 1024) : sdesc_sw64(ka + off, 16, 512);
              mma_ss_f8(tmem + C::col_s(i), da, db, kIdescS8, kk > 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * C::kSubBytes + (kk & 3) * 32;
              mma_ss(tmem + C::col_s(i), sdesc_sw128(qa + off, 16, 1024),
                     sdesc_sw128(ka + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars->s_full[i]);
        }
        __syncwarp();
      };
      int g = 0, qn = 0;
      int ns[2] = {0, 0};   // S_i issued so far
      bool ok = true;
      for (int r = 0; ok && r * grid < p.total_units; ++r) {
        const int L = unit_index(r, cta, grid);
        if (L >= p.total_units) continue;
        const Unit u = unit_of<CAUSAL, GEN>(p, L);
        const int qb = qn % C::kQBufs;
        if (!wait_w(&bars->q_full[qb], (qn / C::kQBufs) & 1, wc)) { ok = false; break; }
        UnitSteps<CAUSAL, GEN> us;
        if constexpr (GEN) us.begin(p, u);
        for (int j = 0; j < u.n_steps; ++j, ++g) {
          if constexpr (GEN) us.next(u, j);
          const int st = g % C::kStages;
          if (!wait_w(&bars->k_full[st], (g / C::kStages) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (GEN ? !us.act[i] : j >= u.nkv[i]) continue;
            if (ns[i] > 0) {
              // S_i may be overwritten once its softmax has read it (P in its own columns)
              // or, when P_i lives in S_i's columns, once P_i·V has consumed P_i.
              uint64_t* freed = C::kSepP ? &bars->s_free[i] : &bars->pv_done[i];
              if (!wait_w(freed, (ns[i] - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after_sync();
            }
            issue_s(qb, i, st);
            ++ns[i];
            FA_TRACE(16 + i, j);
          }
          if (!ok) break;
          commit(&bars->kv_empty[st]);  // K_j is free once these S MMAs are done
        }
        if (!ok) break;
        commit(&bars->q_empty[qb]);     // this unit's Q is free once its S MMAs are done
        ++qn;
      }
    } else {
      // O_i += P_i · V_st : A = P from TMEM (8 columns = 16 keys per step), B = V tile,
      // MN-major (D contiguous): 16 keys = 2048 bytes per step; next 64-wide column block
      // (leading byte offset) 16 KB away; next 8-key group (stride byte offset) 1 KB away.
      // Issued in C::kPParts parts of the keys as the softmax stores them; part h < last is
      // committed to pv_part[i][h], the whole to pv_done[i].
      constexpr uint32_t kIdescO = idesc_bf16(kBlockM, D, true);
      const uint32_t v_base = smem_u32(smem + C::kVOff);
      auto issue_pv = [&](int i, int st, bool acc, int h) {
        if (leader) {
          const uint32_t va = v_base + st * C::kTileBytes;
          constexpr int kPer = kBlockN / 16 / C::kPParts;  // K = 16 steps per part
#pragma unroll
          for (int k4 = 0; k4 < kPer; ++k4) {
            const int kk = h * kPer + k4;
            mma_ts(tmem + C::col_o(i), tmem + C::col_p(i) + kk * 8,
                   sdesc_sw128(va + kk * 2048, C::kSubBytes, 1024), kIdescO,
                   (acc || kk > 0) ? 1u : 0u);
          }
          mma_commit(h == C::kPParts - 1 ? &bars->pv_done[i] : &bars->pv_part[i][h]);
        }
        __syncwarp();
      };
      int g = 0;
      int np[2] = {0, 0};       // P_i·V issued so far
      int nunits[2] = {0, 0};   // finished units in which tile i was active
      bool ok = true;
      for (int r = 0; ok && r * grid < p.total_units; ++r) {
        const int L = unit_index(r, cta, grid);
        if (L >= p.total_units) continue;
        const Unit u = unit_of<CAUSAL, GEN>(p, L);
        UnitSteps<CAUSAL, GEN> us;
        if constexpr (GEN) us.begin(p, u);
        int jt[2] = {0, 0};   // steps of this unit in which tile i was active
        for (int j = 0; j < u.n_steps; ++j, ++g) {
          if constexpr (GEN) us.next(u, j);
          const int st = g % C::kStages;
          if (!wait_w(&bars->v_full[st], (g / C::kStages) & 1, wc)) { ok = false; break; }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (GEN ? !us.act[i] : j >= u.nkv[i]) continue;
            if (jt[i] == 0 && nunits[i] > 0) {
              // This unit's first P·V overwrites O_i: the previous unit's O_i must have
              // been read out.
              if (!wait_w(&bars->o_free[i], (nunits[i] - 1) & 1, wc)) { ok = false; break; }
            }
#pragma unroll
            for (int h = 0; h < C::kPParts; ++h) {
              if (!wait_w(&bars->p_full[i][h], np[i] & 1, wc)) { ok = false; break; }
              if (h == 0) FA_TRACE(11 + i, j);
              tc_fence_after_sync();
              issue_pv(i, st, jt[i] > 0, h);
            }
            if (!ok) break;
            ++np[i];
            ++jt[i];
            FA_TRACE(14 + i, j);
          }
          if (!ok) break;
          commit(&bars->kv_empty[st]);  // V_j is free once these P·V MMAs are done
        }
#pragma unroll
        for (int i = 0; i < 2; ++i)
          if (u.nkv[i] > 0) ++nunits[i];
      }
    }
    // Nothing may still be running on the tensor core when TMEM is released.
    commit(&bars->mma_done);
    wait_w(&bars->mma_done, 0, drain);
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int wg = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::col_s(wg);
    const uint32_t t_o = tmem + lane_off + C::col_o(wg);
    const uint32_t t_p = tmem + lane_off + C::col_p(wg);
    const float c = p.scale_log2;

    int gs = 0;     // S_i consumed (= P_i produced) so far over this CTA's units
    bool ok = true;
    // Where a unit's rows go: the bf16 output (row_idx; r0 = the warp's first row, for the
    // TMA store) and LSE, or (general form with several key ranges) the fp32 partial row
    // and LSE of its range.
    struct RowOut {
      size_t row_idx, part_idx;
      int r0, bh;
      bool in_range, partial;
    };
    // Writes 32 output columns from c0 directly: fp32 scaled by mul (partial) or bf16.
    auto write_row = [&](const RowOut& w, const uint32_t* r, int c0, float mul) {
      if (!w.in_range) return;
      if (w.partial) {
        float4* prow = reinterpret_cast<float4*>(p.o_part + w.part_idx * D + c0);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          prow[t] = make_float4(u2f(r[4 * t]) * mul, u2f(r[4 * t + 1]) * mul,
                                u2f(r[4 * t + 2]) * mul, u2f(r[4 * t + 3]) * mul);
      } else {
        uint4* orow = reinterpret_cast<uint4*>(p.o + w.row_idx * D);
        uint32_t ob[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) ob[t] = pack_bf16x2(u2f(r[2 * t]) * mul, u2f(r[2 * t + 1]) * mul);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          orow[c0 / 8 + t] = make_uint4(ob[4 * t], ob[4 * t + 1], ob[4 * t + 2], ob[4 * t + 3]);
      }
    };
    auto write_lse = [&](const RowOut& w, float v) {
      if (!w.in_range) return;
      if (w.partial) p.lse_part[w.part_idx] = v;
      else p.lse[w.row_idx] = v;
    };
    // A row that saw no key (general form: O = 0, LSE = −∞) or a failed unit (NaN).
    auto write_const_row = [&](const RowOut& w, uint32_t bits) {
      if (!w.in_range) return;
      if (w.partial) {
        float4* prow = reinterpret_cast<float4*>(p.o_part + w.part_idx * D);
        const float f = u2f(bits);
#pragma unroll
        for (int t = 0; t < D / 4; ++t) prow[t] = make_float4(f, f, f, f);
      } else {
        uint4* orow = reinterpret_cast<uint4*>(p.o + w.row_idx * D);
        const uint32_t b2 = pack_bf16x2(u2f(bits), u2f(bits));
#pragma unroll
        for (int t = 0; t < D / 8; ++t) orow[t] = make_uint4(b2, b2, b2, b2);
      }
    };
    auto fail_rows = [&](const RowOut& w) {
      write_const_row(w, 0x7FC00000u);
      write_lse(w, __uint_as_float(0x7FC00000u));
    };
    auto lse_of = [&](float l, float m) {
      return (GEN && !(l > 0.0f)) ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
    };
    auto inv_of = [&](float l) { return (GEN && !(l > 0.0f)) ? 0.0f : 1.0f / l; };
    // O_i, already read into registers (D = 64), to the output: each warp stages its 32
    // rows in its own 4 KB slice, 16-byte chunk c of row r at position c ^ (r mod 8) (the
    // map's 128-byte swizzle; conflict-free), and its lane 0 stores them as one 64 × 32
    // box; rows past the sequence are not written. The warp's previous store from the
    // slice (one unit back) must have read it out first.
    auto store_o = [&](const RowOut& w, const uint32_t* o, float l, float m) {
      const float inv_l = inv_of(l);
      if (D == 64 && !w.partial) {
        uint8_t* slice = smem + C::kOOff + (wg * 4 + quad) * 4096;
        const uint32_t ob = smem_u32(slice) + lane * 128;
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < D / 8; ++ch)
          st_shared_v4(ob + ((ch ^ (lane & 7)) << 4),
                       pack_bf16x2(u2f(o[8 * ch]) * inv_l, u2f(o[8 * ch + 1]) * inv_l),
                       pack_bf16x2(u2f(o[8 * ch + 2]) * inv_l, u2f(o[8 * ch + 3]) * inv_l),
                       pack_bf16x2(u2f(o[8 * ch + 4]) * inv_l, u2f(o[8 * ch + 5]) * inv_l),
                       pack_bf16x2(u2f(o[8 * ch + 6]) * inv_l, u2f(o[8 * ch + 7]) * inv_l));
        fence_proxy_async_smem();  // the staged rows, visible to the TMA engine
        __syncwarp();
        if (lane == 0 && w.r0 < p.T) {
          tma_store_3d(&tm_o, slice, 0, w.r0, w.bh);
          bulk_commit_group();
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) write_row(w, o + c0, c0, inv_l);
      }
      write_lse(w, lse_of(l, m));
    };
    // Reads O_i (after its last P·V) into registers and releases it to the next unit's
    // first P·V.
    auto read_o = [&](uint32_t* o) {
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) tmem_ld32(t_o + c0, o + c0);
      tmem_ld_wait();
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) reg_fence32(o + c0);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[wg]);
    };
    // D = 64 defers a unit's epilogue into this tile's first step of its next unit: that
    // step's S load, max and exponentials run while the unit's last P·V finishes, its P is
    // stored as soon as that P·V is done, and only then is O read out and written. (Run
    // at once, the epilogue and the next unit's set-up, code that runs once per unit, sat
    // between the two P·V products on the tensor core.) D = 128 keeps it immediate: its
    // O would need 128 more registers.
    // The pending unit's l, m and output position wait in shared memory (this thread's
    // 16-byte record), not in registers the step loop needs. The fp32 partial rows of the
    // general form keep the immediate epilogue.
    const bool defer = C::kDefer && !(GEN && p.n_splits > 1);
    bool pend = false;
    float4* const prec = reinterpret_cast<float4*>(smem + C::kPendOff) + wg * kBlockM + row;
    auto park = [&](const RowOut& w, float l, float m) {
      *prec = make_float4(l, m, __int_as_float(w.r0), __int_as_float(w.bh));
      pend = true;
    };
    auto parked = [&](float& l, float& m) {
      const float4 v = *prec;
      l = v.x;
      m = v.y;
      const int r0 = __float_as_int(v.z), bh = __float_as_int(v.w);
      const int q_row = r0 + lane;
      return RowOut{static_cast<size_t>(bh) * static_cast<size_t>(p.T) + static_cast<size_t>(q_row),
                    0, r0, bh, q_row < p.T, false};
    };
    auto fail_pending = [&]() {
      float l, m;
      fail_rows(parked(l, m));
      pend = false;
    };
    // Finishes the pending unit once its last P·V is done (already waited for when
    // `waited`).
    auto flush_pending = [&](bool waited) {
      const bool good = waited || (ok && wait_w(&bars->pv_done[wg], (gs - 1) & 1, wc));
      if (good) {
        if (!waited) tc_fence_after_sync();
        uint32_t o[D];
        read_o(o);
        float l, m;
        const RowOut w = parked(l, m);
        store_o(w, o, l, m);
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
      // (ternaries, not u.nkv[wg]: a runtime index would move the unit to local memory)
      const int n = wg ? u.nkv[1] : u.nkv[0];
      const int qt = u.qt0 + wg;
      const int q_row = qt * kBlockM + row;
      const bool tile_exists = wg < p.tiles_per_cta && qt * kBlockM < p.T;
      if (n == 0 && !(GEN && tile_exists)) continue;
      const RowOut cur{static_cast<size_t>(u.bh) * static_cast<size_t>(p.T) +
                           static_cast<size_t>(q_row),
                       (static_cast<size_t>(u.split) * p.BH + u.bh) * static_cast<size_t>(p.T) +
                           q_row,
                       qt * kBlockM + quad * 32, u.bh, q_row < p.T, GEN && p.n_splits > 1};
      if (!ok) {
        // A wait gave up earlier: mark every row this warpgroup owns as failed.
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      if (n == 0) {  // general form: this tile uses no K tile of the range
        if (pend) flush_pending(false);
        write_const_row(cur, 0u);
        write_lse(cur, -INFINITY);
        continue;
      }

      float m_ref = -INFINITY;  // reference max (base-2 scaled units) shared by O and l
      float l = 0.0f;
      // this tile's K tiles (GEN: its walk, the next position fetched a step ahead)
      Walk w{nullptr, 0};
      int nx = 0;
      if constexpr (GEN) {
        w = walk_of<CAUSAL>(p, u, wg);
        nx = walk_next(w, u.kb - 1);
      }
      int kt = u.kb - 1;  // (dense: u.kb = 0, step j is K tile j)
      for (int j = 0; j < n; ++j, ++gs) {
        if constexpr (GEN) {
          kt = nx;
          nx = walk_next(w, kt);
        } else {
          ++kt;
        }
        if (!wait_w(&bars->s_full[wg], gs & 1, wc)) { ok = false; break; }
        FA_TRACE(30 + wg, j);
        tc_fence_after_sync();
        const int k0 = kt * kBlockN;
        // Keys past the end of the sequence, and (causal) keys after this query.
        int lim;
        bool masked;
        if constexpr (GEN) {
          lim = (CAUSAL ? min(q_row + 1 + p.kv_off, p.Tk) : p.Tk) - k0;
          masked = lim < kBlockN;
        } else {
          lim = (CAUSAL ? min(q_row + 1, p.T) : p.T) - k0;
          masked = (CAUSAL && kt == qt) || (k0 + kBlockN > p.T);
        }

        // S into registers. D = 64: all four 32-column loads in flight before one wait (one
        // TMEM round trip). D = 128: in two halves, the second loading while the first is
        // masked and maxed (measured faster there).
        uint32_t s[kBlockN];
        float mx[8];
        if constexpr (D == 64) {
          tmem_ld32(t_s + 0, s);
          tmem_ld32(t_s + 32, s + 32);
          tmem_ld32(t_s + 64, s + 64);
          tmem_ld32(t_s + 96, s + 96);
          tmem_ld_wait();
          reg_fence32(s);
          reg_fence32(s + 32);
          reg_fence32(s + 64);
          reg_fence32(s + 96);
          if constexpr (C::kSepP) {
            // S_i is in registers: the tensor core may overwrite it with the next S_i.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->s_free[wg]);
          }
          FA_TRACE(20 + wg, j);
          if (masked) {
#pragma unroll
            for (int t = 0; t < kBlockN; ++t)
              if (t >= lim) s[t] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int a = 0; a < 8; ++a) mx[a] = fmaxf(u2f(s[2 * a]), u2f(s[2 * a + 1]));
#pragma unroll
          for (int t = 16; t < kBlockN; t += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], u2f(s[t + 2 * a]), u2f(s[t + 2 * a + 1]));
        } else {
          tmem_ld32(t_s + 0, s);
          tmem_ld32(t_s + 32, s + 32);
          tmem_ld_wait();
          reg_fence32(s);
          reg_fence32(s + 32);
          tmem_ld32(t_s + 64, s + 64);
          tmem_ld32(t_s + 96, s + 96);
          if (masked) {
#pragma unroll
            for (int t = 0; t < 64; ++t)
              if (t >= lim) s[t] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int a = 0; a < 8; ++a) mx[a] = fmaxf(u2f(s[2 * a]), u2f(s[2 * a + 1]));
#pragma unroll
          for (int t = 16; t < 64; t += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], u2f(s[t + 2 * a]), u2f(s[t + 2 * a + 1]));
          tmem_ld_wait();
          reg_fence32(s + 64);
          reg_fence32(s + 96);
          FA_TRACE(20 + wg, j);
          if (masked) {
#pragma unroll
            for (int t = 64; t < kBlockN; ++t)
              if (t >= lim) s[t] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int t = 64; t < kBlockN; t += 16)
#pragma unroll
            for (int a = 0; a < 8; ++a) mx[a] = fmax3(mx[a], u2f(s[t + 2 * a]), u2f(s[t + 2 * a + 1]));
        }
        const float m_tile =
            fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * c;
        FA_TRACE(40 + wg, j);

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
        bool waited = false;

        // p = 2^(s·c − m_ref) on fp32 pairs; row sum in fp32; P kept as bf16 pairs. Each
        // part of the keys is stored and signalled as soon as it is ready.
        const uint64_t c2 = f2_pack(c, c);
        // (general form: a row with no visible key so far keeps m_ref = −∞; its p are 0)
        const float m_use = (GEN && m_ref == -INFINITY) ? 0.0f : m_ref;
        const uint64_t nm2 = f2_pack(-m_use, -m_use);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
        constexpr int kPk = kBlockN / 2 / C::kPParts;  // bf16 pairs per part
#pragma unroll
        for (int h = 0; h < C::kPParts; ++h) {
          uint32_t pk[kPk];
#pragma unroll
          for (int t2 = 0; t2 < kPk; ++t2) {
            const int t = h * kPk + t2;
            const uint64_t x2 = f2_fma(f2_pack(u2f(s[2 * t]), u2f(s[2 * t + 1])), c2, nm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            if (t & 1) acc1 = f2_add(acc1, f2_pack(p0, p1));
            else acc0 = f2_add(acc0, f2_pack(p0, p1));
            pk[t2] = pack_bf16x2(p0, p1);
          }
          if (h == C::kPParts - 1) FA_TRACE(42 + wg, j);
          if (h == 0 && any_rescale) {
            // Rows whose max jumped bring their accumulated O to the new reference (rare:
            // the reference moves only by more than τ), before any of this step's P·V. O
            // must be stable: the previous P·V done. 16 columns at a time (the second half
            // of S may still be live).
            if (C::kSepP && gs > 0) {
              if (!wait_w(&bars->pv_done[wg], (gs - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after_sync();
              waited = true;
            }
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 16) {
              uint32_t r[16];
              tmem_ld16(t_o + c0, r);
              tmem_ld_wait();
              reg_fence16(r);
#pragma unroll
              for (int t = 0; t < 16; ++t) r[t] = __float_as_uint(u2f(r[t]) * alpha);
              tmem_st16(t_o + c0, r);
            }
          }
          if constexpr (C::kSepP) {
            // These P_i columns are free once the matching part of the previous P_i·V is done.
            if (gs > 0 && !waited) {
              if (!wait_w(h == C::kPParts - 1 ? &bars->pv_done[wg] : &bars->pv_part[wg][h],
                                  (gs - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after_sync();
            }
          }
          if constexpr (kPk >= 32) {
#pragma unroll
            for (int c0 = 0; c0 < kPk; c0 += 32) tmem_st32(t_p + h * kPk + c0, pk + c0);
          } else {
            tmem_st16(t_p + h * kPk, pk);
          }
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->p_full[wg][h]);
        }
        if (!ok) break;
        {
          float a0, a1, b0, b1;
          f2_unpack(acc0, a0, a1);
          f2_unpack(acc1, b0, b1);
          l += (a0 + b0) + (a1 + b1);
        }
        FA_TRACE(22 + wg, j);
        // (j = 0) The previous unit's last P·V was the one waited for above: its O_i is
        // final. Read it out (releasing O_i to this unit's first P·V), then write it.
        if (C::kDefer && pend) flush_pending(true);
      }
      if (!ok) {
        if (pend) fail_pending();
        fail_rows(cur);
        continue;
      }
      if (defer) {
        park(cur, l, m_ref);
        continue;
      }

      // Epilogue at once (D = 128, and the partial rows): O / l and the logsumexp, once this
      // unit's last P·V is done.
      const bool good = wait_w(&bars->pv_done[wg], (gs - 1) & 1, wc);
      FA_TRACE(24 + wg, 0);
      if (good) {
        tc_fence_after_sync();
        const float inv_l = inv_of(l);
        if (!cur.partial) {
          // 64 columns per round through the warp's staging slice, 32 at a time from TMEM.
          uint8_t* slice = smem + C::kOOff + (wg * 4 + quad) * 4096;
          const uint32_t ob = smem_u32(slice) + lane * 128;
#pragma unroll 1
          for (int hb = 0; hb < D / 64; ++hb) {
            if (lane == 0) bulk_wait_group_read0();  // the slice's previous store read it
            __syncwarp();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t o[32];
              tmem_ld32(t_o + hb * 64 + half * 32, o);
              tmem_ld_wait();
              reg_fence32(o);
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const int ch = half * 4 + t;
                st_shared_v4(ob + ((ch ^ (lane & 7)) << 4),
                             pack_bf16x2(u2f(o[8 * t]) * inv_l, u2f(o[8 * t + 1]) * inv_l),
                             pack_bf16x2(u2f(o[8 * t + 2]) * inv_l, u2f(o[8 * t + 3]) * inv_l),
                             pack_bf16x2(u2f(o[8 * t + 4]) * inv_l, u2f(o[8 * t + 5]) * inv_l),
                             pack_bf16x2(u2f(o[8 * t + 6]) * inv_l, u2f(o[8 * t + 7]) * inv_l));
              }
            }
            if (hb == D / 64 - 1) {
              // O_i has been read: the next unit's first P·V may overwrite it.
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars->o_free[wg]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && cur.r0 < p.T) {
              tma_store_3d(&tm_o, slice, hb * 64, cur.r0, cur.bh);
              bulk_commit_group();
            }
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(t_o + c0, r);
            tmem_ld_wait();
            reg_fence32(r);
            write_row(cur, r, c0, inv_l);
          }
          // O_i has been read: the next unit's first P·V may overwrite it.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->o_free[wg]);
        }
        write_lse(cur, lse_of(l, m_ref));
        FA_TRACE(26 + wg, 0);
      } else {
        ok = false;
        fail_rows(cur);
      }
    }
    if (pend) flush_pending(false);  // the last unit's epilogue
    // The output rows' TMA stores must have read their shared-memory source before the
    // CTA exits (their global writes complete with the grid).
    if (lane == 0) bulk_wait_group_read0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the key-range partial results of the general form: with M = max_s LSE_s and
// w_s = exp(LSE_s − M), O = Σ w_s·O_s / Σ w_s (bf16) and LSE = M + ln Σ w_s; a row that no
// range saw gets O = 0 and LSE = −∞. This is the merge of results over disjoint key blocks
// that the first FlashAttention's outer K/V loop needed ("手写 FlashAttention", step ③),
// used here to spread one query tile's keys over several CTAs. rows = B·H·Tq.
//
// One warp per row (grid-stride over rows), lane l owning columns l·D/32 … (l+1)·D/32 − 1.
// The lanes read the ranges' LSEs side by side and agree on M and Σ w_s with shuffles; the
// partial rows are then read eight ranges at a time, all loads in flight together. The
// merge sits between a kernel and the caller's next one, so its latency, not its bytes,
// is what it costs.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_combine_kernel(const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part,
                                                             __nv_bfloat16* __restrict__ o,
                                                             float* __restrict__ lse,
                                                             int n_splits, int rows) {
  constexpr int C = D / 32;  // columns per lane: 2 or 4
  // Launched as a programmatic dependent of the kernel that wrote the partials.
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    float m = -INFINITY;
    for (int s = lane; s < n_splits; s += 32)
      m = fmaxf(m, lse_part[static_cast<size_t>(s) * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int base = 0; base < n_splits; base += 32) {
        const int cnt = min(32, n_splits - base);
        // lane l: the weight of range base + l (0 for a range that saw no key)
        float wl = 0.f;
        if (lane < cnt) {
          const float ls = lse_part[static_cast<size_t>(base + lane) * rows + row];
          wl = (ls == -INFINITY) ? 0.f : expf(ls - m);
        }
        wsum += wl;
        const float* src = o_part + (static_cast<size_t>(base) * rows + row) * D + lane * C;
        const size_t step = static_cast<size_t>(rows) * D;
        for (int j0 = 0; j0 < cnt; j0 += 8) {
          float x[8][C];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j0 + j < cnt) {
              if constexpr (C == 2) {
                const float2 t = *reinterpret_cast<const float2*>(src + (j0 + j) * step);
                x[j][0] = t.x;
                x[j][1] = t.y;
              } else {
                const float4 t = *reinterpret_cast<const float4*>(src + (j0 + j) * step);
                x[j][0] = t.x;
                x[j][1] = t.y;
                x[j][2] = t.z;
                x[j][3] = t.w;
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float w = __shfl_sync(0xffffffffu, wl, (j0 + j) & 31);
            if (j0 + j < cnt) {
#pragma unroll
              for (int c = 0; c < C; ++c) acc[c] = fmaf(w, x[j][c], acc[c]);
            }
          }
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* dst = o + static_cast<size_t>(row) * D + lane * C;
    if constexpr (C == 2) {
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    } else {
      uint2 out;
      out.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      out.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(dst) = out;
    }
    if (lane == 0) lse[row] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

}  // namespace fa
