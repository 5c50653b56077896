"""Plain, slow fp64 oracle for scaled-dot-product attention (forward and backward).

TEST INFRASTRUCTURE ONLY: never imported by the product path.

What is computed, per (batch b, head h), for query rows i and key rows j of one
sequence of length T (the naive form that [HW-FA] step ① writes out as
S = QKᵀ/√d → softmax → P·V, and [KCS] "注意力算法" draws):

    S[i, j]  = scale · q_i · k_j                      (scale = 1/√d in every workload)
    S[i, j]  = −∞           where causal and j > i    ([HW-FA] step ③: the upper-right
                                                       part of the score grid is masked)
    m_i      = max_j S[i, j]                          (safe softmax: [HW-FA] step ②
                                                       "why subtract the max",
                                                       [KCS] "指数中的数值稳定性")
    P[i, j]  = exp(S[i, j] − m_i) / Σ_j exp(S[i, j] − m_i)
    O_i      = Σ_j P[i, j] · v_j
    LSE_i    = m_i + ln Σ_j exp(S[i, j] − m_i)        (the per-row logsumexp that
                                                       [HW-FA] step ④ says the forward
                                                       keeps for the backward pass;
                                                       natural log of the scaled scores)

Inputs are upcast exactly to fp64 (bf16 → fp64 is exact) and every step runs in fp64
with numpy; matrix products use numpy's BLAS. Nothing is tiled and there is no online
recurrence here: the whole score row of a query is materialised. Rows are processed
in chunks only to bound memory, and each row's result depends on that row alone, so
chunking changes no arithmetic.

The scalar online recurrence of [HW-FA] step ② (running max m, running sum l rescaled
by exp(m_old − m_new), accumulator rescaled by the same factor, one final ÷l) is given
separately by :func:`online_softmax_trace` and :func:`online_weighted_sum`, so that the
tests can pin the recurrence itself against the one-pass definition.

The backward pass (:func:`attention_backward`) is the derivative of that same definition
with respect to Q, K and V for an upstream gradient dO, written out by the chain rule:

    dV = Pᵀ·dO,   dP = dO·Vᵀ,   dS_ij = P_ij·(dP_ij − Σ_k P_ik·dP_ik),
    dQ = scale·dS·K,   dK = scale·dSᵀ·Q.

[HW-FA] step ④ (its part on training) says the forward keeps only the per-row
logsumexp so that the backward can recompute S and P block by block, and [FA-tiling]
§2.2 (FlashAttention core ideas, ijyty.com: backward recomputation, per-block gradients
summed into the global gradient). Neither page prints a backward formula, so this is the
plain derivative, evaluated naively on the whole score row.

Pinned by ``tests/test_oracle.py`` (closed forms, invariants, brute force, finite
differences and planted-mistake checks); nothing here is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

# Rows of S materialised at once; a chunk of 512 rows at T = 16384 is 64 MB of fp64.
_ROW_CHUNK = 512


def _as_f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Steps of the definition. Each is a separate function so that the tests can plant a
# mistake in exactly one step and check that some pin catches it.
# --------------------------------------------------------------------------------------

def scores(q_rows: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale · Q Kᵀ for the given query rows ([HW-FA] step ①). Shapes [R,d],[T,d] → [R,T]."""
    return scale * (q_rows @ k.T)


def apply_causal_mask(s: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """Set S[r, j] = −∞ where key j lies after query row rows[r] ([HW-FA] step ③).

    Key j is visible to query i iff j ≤ i. Query and key sequences have the same
    length here, so top-left and bottom-right alignment of the mask coincide.
    """
    T = s.shape[1]
    j = np.arange(T)[None, :]
    return np.where(j > rows[:, None], -np.inf, s)


def safe_softmax(s: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Row-wise softmax with the row max subtracted first ([HW-FA] step ②; [KCS] safe softmax).

    Returns (P, m, l): the probabilities, the row max m and the row sum
    l = Σ_j exp(S[i,j] − m_i). Every exponent is ≤ 0, so nothing overflows.
    """
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    return e / l, m[:, 0], l[:, 0]


def weighted_values(p: np.ndarray, v: np.ndarray) -> np.ndarray:
    """O = P · V ([HW-FA] step ①, the last product of the naive form)."""
    return p @ v


def logsumexp_from(m: np.ndarray, l: np.ndarray) -> np.ndarray:
    """LSE_i = m_i + ln l_i, natural log of Σ_j exp(S[i,j]) ([HW-FA] step ④ on the backward pass)."""
    return m + np.log(l)


# --------------------------------------------------------------------------------------
# Public entry points.
# --------------------------------------------------------------------------------------

def attention_rows(q, k, v, causal: bool, scale: float, rows) -> tuple[np.ndarray, np.ndarray]:
    """O and LSE for selected query rows of ONE (batch, head).

    q, k, v: [T, d] arrays (any real dtype; upcast to fp64). rows: 1-D int array of
    query indices in [0, T). Returns (O [R, d] fp64, LSE [R] fp64).
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    rows = np.asarray(rows, dtype=np.int64)
    s = scores(q[rows], k, scale)
    if causal:
        s = apply_causal_mask(s, rows)
    p, m, l = safe_softmax(s)
    return weighted_values(p, v), logsumexp_from(m, l)


def attention(q, k, v, causal: bool, scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Exact attention forward for all heads.

    q, k, v: [B, H, T, d] arrays. Returns (O [B,H,T,d] fp64, LSE [B,H,T] fp64).
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    B, H, T, d = q.shape
    o = np.empty((B, H, T, d), dtype=np.float64)
    lse = np.empty((B, H, T), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, T, _ROW_CHUNK):
                rows = np.arange(r0, min(T, r0 + _ROW_CHUNK))
                o[b, h, rows], lse[b, h, rows] = attention_rows(
                    q[b, h], k[b, h], v[b, h], causal, scale, rows)
    return o, lse


# --------------------------------------------------------------------------------------
# The online recurrence, as [HW-FA] step ② states it, for pinning the recurrence.
# --------------------------------------------------------------------------------------

def online_softmax_trace(x, block: int):
    """Read the scores ``x`` ``block`` at a time, keeping only m and l ([HW-FA] step ②).

    m is the largest score read so far and l = Σ exp(x − m) over the scores read so
    far, taken relative to the current m. When a block raises the max, the old l is
    multiplied by alpha = exp(m_old − m_new) before the block's own terms are added.

    Returns a list with one tuple per block: (scores read, m, l, alpha). At the first
    block alpha is exp(−∞) = 0. softmax(x) = exp(x − m_last) / l_last.
    """
    x = [float(t) for t in x]
    m = -math.inf
    l = 0.0
    trace = []
    for start in range(0, len(x), block):
        xb = x[start:start + block]
        m_new = max(m, max(xb))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        l = l * alpha + sum(math.exp(t - m_new) for t in xb)
        m = m_new
        trace.append((start + len(xb), m, l, alpha))
    return trace


def online_weighted_sum(x, vals, block: int):
    """softmax(x) · vals by the blocked recurrence of [HW-FA] step ②.

    acc holds Σ exp(x − m)·v relative to the m current when each term was added;
    when the max rises, acc and l are both multiplied by the same
    alpha = exp(m_old − m_new); after the last block the result is acc / l (the
    division done once, at the end). ``vals`` is [n, d].
    """
    x = np.asarray(x, dtype=np.float64)
    vals = np.asarray(vals, dtype=np.float64)
    m = -np.inf
    l = 0.0
    acc = np.zeros(vals.shape[1], dtype=np.float64)
    for start in range(0, x.shape[0], block):
        xb = x[start:start + block]
        m_new = max(m, float(xb.max()))
        alpha = math.exp(m - m_new) if m != -np.inf else 0.0
        p = np.exp(xb - m_new)
        l = l * alpha + float(p.sum())
        acc = acc * alpha + p @ vals[start:start + block]
        m = m_new
    return acc / l, m, l


# --------------------------------------------------------------------------------------
# Backward pass: the derivative of the forward definition.
# --------------------------------------------------------------------------------------

def grad_values(p: np.ndarray, do_rows: np.ndarray) -> np.ndarray:
    """dV contribution of these query rows: Pᵀ·dO (O = P·V is linear in V)."""
    return p.T @ do_rows


def grad_probs(do_rows: np.ndarray, v: np.ndarray) -> np.ndarray:
    """dP = dO·Vᵀ."""
    return do_rows @ v.T


def softmax_backward(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """dS = P ∘ (dP − rowsum(P ∘ dP)): the Jacobian of a softmax row applied to dP
    (masked entries have P = 0 and get dS = 0)."""
    return p * (dp - np.sum(p * dp, axis=1, keepdims=True))


def grad_queries(ds: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """dQ rows = scale·dS·K (S = scale·Q·Kᵀ)."""
    return scale * (ds @ k)


def grad_keys(ds: np.ndarray, q_rows: np.ndarray, scale: float) -> np.ndarray:
    """dK contribution of these query rows: scale·dSᵀ·Q."""
    return scale * (ds.T @ q_rows)


def attention_backward_head(q, k, v, do, causal: bool, scale: float, row_chunk: int = 512):
    """(dQ, dK, dV) of one (batch, head); q, k, v, do: [T, d]. Query rows are taken in
    chunks; each chunk's terms are exact and dK, dV are sums over query rows."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(do)
    T = q.shape[0]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, T, row_chunk):
        rows = np.arange(r0, min(T, r0 + row_chunk))
        s = scores(q[rows], k, scale)
        if causal:
            s = apply_causal_mask(s, rows)
        p, _, _ = safe_softmax(s)
        dv += grad_values(p, do[rows])
        ds = softmax_backward(p, grad_probs(do[rows], v))
        dq[rows] = grad_queries(ds, k, scale)
        dk += grad_keys(ds, q[rows], scale)
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, causal: bool, scale: float, rows):
    """dQ of the given query rows only (one head; [T, d] inputs). Each dQ row needs only
    its own row of P and dP, so sampled rows can be checked at any T."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(do)
    rows = np.asarray(rows)
    s = scores(q[rows], k, scale)
    if causal:
        s = apply_causal_mask(s, rows)
    p, _, _ = safe_softmax(s)
    ds = softmax_backward(p, grad_probs(do[rows], v))
    return grad_queries(ds, k, scale)


def attention_backward_cols(q, k, v, do, causal: bool, scale: float, cols,
                            row_chunk: int = 512):
    """dK and dV of the given key rows only (one head): each needs one column of P and dS
    over all query rows, taken here in chunks of query rows."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(do)
    cols = np.asarray(cols)
    T = q.shape[0]
    dk = np.zeros((len(cols), k.shape[1]))
    dv = np.zeros((len(cols), v.shape[1]))
    for r0 in range(0, T, row_chunk):
        rows = np.arange(r0, min(T, r0 + row_chunk))
        s = scores(q[rows], k, scale)
        if causal:
            s = apply_causal_mask(s, rows)
        p, _, _ = safe_softmax(s)
        ds = softmax_backward(p, grad_probs(do[rows], v))
        dv += grad_values(p[:, cols], do[rows])
        dk += grad_keys(ds[:, cols], q[rows], scale)
    return dk, dv


def attention_backward(q, k, v, do, causal: bool, scale: float):
    """Gradients of L = Σ dO ∘ O with respect to q, k, v ([B, H, T, d] arrays, fp64 out)."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(do)
    B, H, T, d = q.shape
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = attention_backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], causal, scale)
    return dq, dk, dv


def attention_backward_magnitudes(q, k, v, do, causal: bool, scale: float,
                                  row_chunk: int = 512):
    """Error-bound magnitudes of the backward's sums, per output element.

    A sum Σ a_j·b_j whose terms each carry a relative error ≤ u is off by at most
    u·Σ|a_j|·|b_j| (the usual floating-point bound). An implementation that rounds P and
    dS to a short format and forms D = Σ_c dO_c·O_c from a rounded O perturbs dS_ij by up
    to u·A_ij with

        A_ij = |dS_ij| + P_ij·Σ_c |dO_ic|·(|O_ic| + |V_jc|)

    (the second term: the rounding of O inside D, and of dP = dO·V_j). So the sums are
    bounded through

        M_dV = Pᵀ·|dO|,   M_dK = scale·Aᵀ·|Q|,   M_dQ = scale·A·|K|.

    Arrays as attention_backward."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    do = _as_f64(do)
    B, H, T, d = q.shape
    mq = np.empty_like(q)
    mk = np.zeros_like(k)
    mv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, T, row_chunk):
                rows = np.arange(r0, min(T, r0 + row_chunk))
                s = scores(q[b, h, rows], k[b, h], scale)
                if causal:
                    s = apply_causal_mask(s, rows)
                p, _, _ = safe_softmax(s)
                o_rows = weighted_values(p, v[b, h])
                ado = np.abs(do[b, h, rows])
                a = np.abs(softmax_backward(p, grad_probs(do[b, h, rows], v[b, h])))
                a += p * (np.sum(ado * np.abs(o_rows), axis=1, keepdims=True)
                          + ado @ np.abs(v[b, h]).T)
                mv[b, h] += p.T @ ado
                mq[b, h, rows] = scale * (a @ np.abs(k[b, h]))
                mk[b, h] += scale * (a.T @ np.abs(q[b, h, rows]))
    return mq, mk, mv


# --------------------------------------------------------------------------------------
# General form: Tq queries over Tk keys, bottom-right causal alignment, block masks, and
# the merge of results computed over disjoint key ranges.
# --------------------------------------------------------------------------------------

def general_mask(Tq: int, Tk: int, causal: bool, block_mask=None, block: int = 128):
    """Boolean [Tq, Tk] visibility. Causal is aligned bottom-right: query i sees key j iff
    j ≤ i + (Tk − Tq) (the last query sees every key, as a new token does against its KV
    cache — [HW-FA] step ①'s note that generation keeps the K/V of all earlier tokens).
    block_mask ([ceil(Tq/block), ceil(Tk/block)], nonzero = keep) switches whole blocks
    off, the tile-skipping generalisation of causal masking in [KCS] "块稀疏注意力 V2 和 V3"."""
    vis = np.ones((Tq, Tk), dtype=bool)
    if causal:
        vis &= np.arange(Tk)[None, :] <= (np.arange(Tq) + (Tk - Tq))[:, None]
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        vis &= bm[np.arange(Tq) // block][:, np.arange(Tk) // block]
    return vis


def attention_general_head(q, k, v, causal: bool, scale: float, block_mask=None,
                           block: int = 128):
    """(O, LSE) of one head for q [Tq, d], k and v [Tk, d] under general_mask. A row that
    sees no key at all has O = 0 and LSE = −∞ (the softmax over an empty set is undefined;
    this is the convention of the library)."""
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    Tq, Tk = q.shape[0], k.shape[0]
    vis = general_mask(Tq, Tk, causal, block_mask, block)
    o = np.zeros((Tq, v.shape[1]))
    lse = np.full(Tq, -np.inf)
    for r0 in range(0, Tq, _ROW_CHUNK):
        rows = np.arange(r0, min(Tq, r0 + _ROW_CHUNK))
        s = scores(q[rows], k, scale)
        s = np.where(vis[rows], s, -np.inf)
        live = vis[rows].any(axis=1)
        if live.any():
            p, m, l = safe_softmax(s[live])
            o[rows[live]] = weighted_values(p, v)
            lse[rows[live]] = logsumexp_from(m, l)
    return o, lse


def attention_general(q, k, v, causal: bool, scale: float, block_mask=None, block: int = 128):
    """[B, H, Tq, d] queries over [B, H, Tk, d] keys/values. block_mask is None, one
    [n_qb, n_kb] array shared by every head, or [B·H, n_qb, n_kb] per head."""
    q = _as_f64(q)
    B, H, Tq, d = q.shape
    o = np.empty((B, H, Tq, v.shape[-1]))
    lse = np.empty((B, H, Tq))
    for b in range(B):
        for h in range(H):
            bm = None
            if block_mask is not None:
                bm = np.asarray(block_mask)
                bm = bm[b * H + h] if bm.ndim == 3 else bm
            o[b, h], lse[b, h] = attention_general_head(q[b, h], k[b, h], v[b, h], causal,
                                                        scale, bm, block)
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Combine results computed over disjoint key ranges (index 0 of each array = range):
    with M = max_s LSE_s, weights w_s = exp(LSE_s − M), O = Σ w_s·O_s / Σ w_s and
    LSE = M + ln Σ w_s. This is the merge [HW-FA] step ③ says the first version's outer
    loop over K/V blocks needed; ranges that saw no key carry LSE = −∞ and weight 0."""
    o_parts = _as_f64(o_parts)
    lse_parts = _as_f64(lse_parts)
    m = np.max(lse_parts, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe[None])
    wsum = np.sum(w, axis=0)
    o = np.sum(w[..., None] * o_parts, axis=0) / np.where(wsum > 0, wsum, 1.0)[..., None]
    lse = np.where(wsum > 0, m_safe + np.log(np.where(wsum > 0, wsum, 1.0)), -np.inf)
    return o, lse
