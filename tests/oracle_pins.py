"""Pins for the CPU oracle: checks that hold by mathematics or by what the pages fix.

Each pin takes the oracle module (so that tests can also run the pins against copies
of the oracle with one planted mistake) and raises AssertionError when it fails.

Pages: [HW-FA] "Hand-written FlashAttention" (learn-llm.fim.ai chapter 19);
[KCS] "Kernel case study: Flash Attention" (cnblogs translation).
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _qkv(seed, B, H, T, d, std=1.0):
    r = _rng(seed)
    return (r.standard_normal((B, H, T, d)) * std, r.standard_normal((B, H, T, d)) * std,
            r.standard_normal((B, H, T, d)) * std)


# ----------------------------------------------------------------------------- brute force

def brute_force(q, k, v, causal, scale):
    """Pure-Python loops with ``math``: the definition, one output element at a time."""
    q = np.asarray(q).tolist()
    k = np.asarray(k).tolist()
    v = np.asarray(v).tolist()
    B, H, T, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    o = [[[[0.0] * d for _ in range(T)] for _ in range(H)] for _ in range(B)]
    lse = [[[0.0] * T for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(T):
                keys = [j for j in range(T) if (not causal) or j <= i]
                s = {j: scale * sum(q[b][h][i][t] * k[b][h][j][t] for t in range(d))
                     for j in keys}
                m = max(s.values())
                e = {j: math.exp(s[j] - m) for j in keys}
                l = sum(e.values())
                for t in range(d):
                    o[b][h][i][t] = sum(e[j] * v[b][h][j][t] for j in keys) / l
                lse[b][h][i] = m + math.log(l)
    return np.array(o), np.array(lse)


# ----------------------------------------------------------------------------- pins

def pin_bruteforce(orc):
    """Tiny shapes: numpy oracle == pure-Python loops within 1e-12."""
    cases = [(1, 1, 1, 1), (1, 2, 5, 3), (2, 1, 9, 4), (2, 2, 7, 2), (1, 1, 8, 4)]
    for n, (B, H, T, d) in enumerate(cases):
        q, k, v = _qkv(100 + n, B, H, T, d, std=1.5)
        for causal in (False, True):
            for scale in (1.0 / math.sqrt(d), 0.37):
                o, lse = orc.attention(q, k, v, causal, scale)
                ob, lb = brute_force(q, k, v, causal, scale)
                assert np.max(np.abs(o - ob)) <= 1e-12, (B, H, T, d, causal, scale)
                assert np.max(np.abs(lse - lb)) <= 1e-12, (B, H, T, d, causal, scale)


def pin_hand_example(orc):
    """T=3, d=1, scale 1, worked by hand.

    q = (1, 0, 2), k = (1, 2, 0), v = (1, 0, 3). Row 0 scores: (1, 2, 0).
    Non-causal row 0: O = (e¹·1 + e²·0 + e⁰·3) / (e¹ + e² + e⁰), LSE = ln(e¹ + e² + 1).
    Causal row 0 sees only key 0: O = 1, LSE = 1. Causal row 2 (q=2): scores (2, 4, 0):
    O = (e²·1 + e⁴·0 + 1·3)/(e² + e⁴ + 1).
    """
    q = np.array([1.0, 0.0, 2.0]).reshape(1, 1, 3, 1)
    k = np.array([1.0, 2.0, 0.0]).reshape(1, 1, 3, 1)
    v = np.array([1.0, 0.0, 3.0]).reshape(1, 1, 3, 1)
    e = math.e
    o, lse = orc.attention(q, k, v, False, 1.0)
    assert abs(o[0, 0, 0, 0] - (e + 3.0) / (e + e * e + 1.0)) <= 1e-14
    assert abs(lse[0, 0, 0] - math.log(e + e * e + 1.0)) <= 1e-14
    o, lse = orc.attention(q, k, v, True, 1.0)
    assert abs(o[0, 0, 0, 0] - 1.0) <= 1e-15 and abs(lse[0, 0, 0] - 1.0) <= 1e-15
    # row 1: q=0 sees keys 0,1 with equal scores 0 → mean of v0, v1
    assert abs(o[0, 0, 1, 0] - 0.5) <= 1e-15 and abs(lse[0, 0, 1] - math.log(2.0)) <= 1e-15
    want = (e ** 2 + 3.0) / (e ** 2 + e ** 4 + 1.0)
    assert abs(o[0, 0, 2, 0] - want) <= 1e-14
    assert abs(lse[0, 0, 2] - math.log(e ** 2 + e ** 4 + 1.0)) <= 1e-14


def pin_row_sums(orc):
    """Every row of P sums to 1 within 1e-12 ([HW-FA] step ②: softmax normalises each row)."""
    r = _rng(7)
    s = r.standard_normal((13, 29)) * 6.0
    s = orc.apply_causal_mask(s, np.arange(13) + 3)
    p, m, l = orc.safe_softmax(s)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 1e-12)
    assert np.all(p >= 0.0)
    assert np.allclose(m, s.max(axis=1), rtol=0, atol=0)


def pin_constant_v(orc):
    """V ≡ c gives O ≡ c, whatever the scores and the mask."""
    q, k, _ = _qkv(11, 2, 2, 37, 8, std=2.0)
    c = np.linspace(-3.0, 5.0, 8)
    v = np.broadcast_to(c, (2, 2, 37, 8)).copy()
    for causal in (False, True):
        o, _ = orc.attention(q, k, v, causal, 0.35)
        assert np.max(np.abs(o - c)) <= 1e-12


def pin_causal_row0(orc):
    """Causal: query 0 sees only key 0, so O₀ = v₀ and LSE₀ = scale·q₀·k₀."""
    q, k, v = _qkv(12, 2, 3, 19, 5)
    scale = 0.61
    o, lse = orc.attention(q, k, v, True, scale)
    assert np.max(np.abs(o[:, :, 0, :] - v[:, :, 0, :])) <= 1e-14
    want = scale * np.einsum("bhd,bhd->bh", q[:, :, 0, :], k[:, :, 0, :])
    assert np.max(np.abs(lse[:, :, 0] - want)) <= 1e-13
    # and the last causal row equals the non-causal result for that row
    o2, lse2 = orc.attention(q, k, v, False, scale)
    assert np.max(np.abs(o[:, :, -1] - o2[:, :, -1])) <= 1e-13
    assert np.max(np.abs(lse[:, :, -1] - lse2[:, :, -1])) <= 1e-13


def pin_uniform(orc):
    """q = 0: all visible scores equal, so O_i is a plain mean of the visible v rows and
    LSE_i = ln(number of visible keys). This pins the LSE base (natural log)."""
    B, H, T, d = 1, 2, 23, 6
    _, k, v = _qkv(13, B, H, T, d)
    q = np.zeros((B, H, T, d))
    o, lse = orc.attention(q, k, v, True, 0.125)
    for i in range(T):
        assert np.max(np.abs(o[:, :, i] - v[:, :, :i + 1].mean(axis=2))) <= 1e-13
        assert np.max(np.abs(lse[:, :, i] - math.log(i + 1))) <= 1e-13
    o, lse = orc.attention(q, k, v, False, 0.125)
    assert np.max(np.abs(o - v.mean(axis=2, keepdims=True))) <= 1e-13
    assert np.max(np.abs(lse - math.log(T))) <= 1e-13


def pin_shift(orc):
    """Adding u to every key adds scale·q_i·u to all of row i's scores: O is unchanged
    and LSE_i moves by exactly that constant."""
    q, k, v = _qkv(14, 1, 2, 31, 4)
    u = np.array([0.5, -1.25, 2.0, 0.75])
    scale = 0.4
    for causal in (False, True):
        o1, l1 = orc.attention(q, k, v, causal, scale)
        o2, l2 = orc.attention(q, k + u, v, causal, scale)
        assert np.max(np.abs(o1 - o2)) <= 1e-12
        assert np.max(np.abs((l2 - l1) - scale * (q @ u))) <= 1e-12


def pin_permutation(orc):
    """Non-causal: permuting the rows of K and V together changes nothing."""
    q, k, v = _qkv(15, 2, 2, 17, 3)
    perm = _rng(16).permutation(17)
    o1, l1 = orc.attention(q, k, v, False, 0.5)
    o2, l2 = orc.attention(q, k[:, :, perm], v[:, :, perm], False, 0.5)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12
    # and O follows the query permutation (rows are independent)
    o3, l3 = orc.attention(q[:, :, perm], k, v, False, 0.5)
    assert np.max(np.abs(o3 - o1[:, :, perm])) <= 1e-12


def pin_large_scores(orc):
    """Scores near ±1000 overflow a plain exp even in fp64 (exp(709.8) is the largest finite
    double); the max-subtracted softmax stays finite ([KCS] "指数中的数值稳定性")."""
    facts = load_page_facts()
    assert facts["fp32_exp_overflow_near"] < 1000.0
    q = np.array([[30.0, -30.0], [31.0, 0.0]]).reshape(1, 1, 2, 2)
    k = np.array([[33.0, 0.0], [0.0, 33.0]]).reshape(1, 1, 2, 2)
    v = np.array([[1.0, 2.0], [3.0, 4.0]]).reshape(1, 1, 2, 2)
    o, lse = orc.attention(q, k, v, False, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    # row 0: scores (990, −990) → P = (1, e^−1980 ≈ 0) → O = v0 and LSE = 990
    assert np.max(np.abs(o[0, 0, 0] - [1.0, 2.0])) <= 1e-15 and abs(lse[0, 0, 0] - 990.0) <= 1e-12
    # row 1: scores (1023, 0) → O = v0, LSE = 1023
    assert np.max(np.abs(o[0, 0, 1] - [1.0, 2.0])) <= 1e-15 and abs(lse[0, 0, 1] - 1023.0) <= 1e-12


def pin_rows_match_full(orc):
    """attention_rows on sampled rows equals the full computation on those rows."""
    q, k, v = _qkv(17, 1, 1, 1100, 8)
    rows = np.array([0, 1, 511, 512, 513, 1023, 1099])
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.3)
        orr, lr = orc.attention_rows(q[0, 0], k[0, 0], v[0, 0], causal, 0.3, rows)
        # BLAS may sum in another order for another row count: equal up to rounding
        assert np.max(np.abs(orr - o[0, 0, rows])) <= 1e-13
        assert np.max(np.abs(lr - lse[0, 0, rows])) <= 1e-13


# ------------------------------------------------------------------ online recurrence pins

def _one_pass(x):
    m = max(x)
    e = [math.exp(t - m) for t in x]
    s = sum(e)
    return [t / s for t in e], m, s


def pin_online_trace(orc):
    """[HW-FA] step ②: 8 scores read 2 at a time, keeping only m and l, end at the
    one-pass max and sum, and the resulting softmax equals the one-pass softmax within
    1e-15. Also 3 at a time (a ragged last block) and a max that jumps in the last block."""
    r = _rng(18)
    cases = [(list(r.standard_normal(8) * 3.0), 2),
             (list(r.standard_normal(8) * 3.0), 3),
             ([0.1, -0.4, 0.3, 0.2, -1.0, 0.0, 0.5, 9.0], 2),
             ([5.0, 4.0, 3.0, 2.0, 1.0, 0.0, -1.0, -2.0], 2)]
    for x, block in cases:
        trace = orc.online_softmax_trace(x, block)
        assert len(trace) == math.ceil(len(x) / block)
        p_ref, m_ref, l_ref = _one_pass(x)
        n, m, l, _ = trace[-1]
        assert n == len(x) and m == m_ref
        assert abs(l - l_ref) <= 1e-15 * l_ref
        p = [math.exp(t - m) / l for t in x]
        assert max(abs(a - b) for a, b in zip(p, p_ref)) <= 1e-15
        # every intermediate state is the one-pass state of the prefix read so far
        prev_m = -math.inf
        for n_read, m_i, l_i, alpha in trace:
            _, mp, lp = _one_pass(x[:n_read])
            assert m_i == mp and abs(l_i - lp) <= 1e-15 * lp
            want_alpha = 0.0 if prev_m == -math.inf else math.exp(prev_m - m_i)
            assert abs(alpha - want_alpha) <= 1e-15
            prev_m = m_i


def pin_online_weighted_sum(orc):
    """acc and l rescaled by the same alpha, one ÷l at the end, equals softmax(x)·V."""
    r = _rng(19)
    for n, block in [(8, 2), (8, 3), (37, 5), (64, 64), (5, 1)]:
        x = r.standard_normal(n) * 4.0
        x[-1] += 12.0        # a late jump of the max
        vals = r.standard_normal((n, 6))
        got, m, l = orc.online_weighted_sum(x, vals, block)
        p, mp, lp = _one_pass(list(x))
        want = np.array(p) @ vals
        assert np.max(np.abs(got - want)) <= 1e-14
        assert m == mp and abs(l - lp) <= 1e-14 * lp


def pin_sdpa_library(orc):
    """Cross-check against PyTorch's CPU scaled_dot_product_attention in fp64 (a library
    routine that computes the same definition)."""
    import torch
    import torch.nn.functional as F
    q, k, v = _qkv(20, 2, 3, 45, 16)
    for causal in (False, True):
        o, _ = orc.attention(q, k, v, causal, 0.25)
        ot = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                            torch.from_numpy(v), is_causal=causal,
                                            scale=0.25).numpy()
        assert np.max(np.abs(o - ot)) <= 1e-12


# ------------------------------------------------------------------ backward-pass pins

def _loss_bruteforce(q, k, v, do, causal, scale):
    """L = Σ dO ∘ O with O from the pure-Python definition."""
    o, _ = brute_force(q, k, v, causal, scale)
    return float(np.sum(np.asarray(do) * o))


def pin_bwd_finite_diff(orc):
    """Every gradient element equals a central difference of L = Σ dO ∘ O, with the
    forward taken from the pure-Python loops (not from the oracle), within 1e-7."""
    cases = [(1, 1, 5, 3, True), (1, 1, 5, 3, False), (1, 2, 4, 2, True)]
    h = 1e-5
    for n, (B, H, T, d, causal) in enumerate(cases):
        q, k, v = _qkv(200 + n, B, H, T, d)
        do = _rng(300 + n).standard_normal((B, H, T, d))
        scale = 0.7
        grads = orc.attention_backward(q, k, v, do, causal, scale)
        for which, g in enumerate(grads):
            base = [q, k, v]
            for idx in np.ndindex(*q.shape):
                plus = [t.copy() for t in base]
                minus = [t.copy() for t in base]
                plus[which][idx] += h
                minus[which][idx] -= h
                fd = (_loss_bruteforce(*plus, do, causal, scale)
                      - _loss_bruteforce(*minus, do, causal, scale)) / (2 * h)
                assert abs(g[idx] - fd) <= 1e-7, (n, which, idx, g[idx], fd)


def pin_bwd_hand_example(orc):
    """T=2, d=1, no mask, worked by hand. With p_i = σ(c·a_i·(k1 − k0)) the weight of key 1
    in row i, O_i = v0 + p_i·(v1 − v0), so for L = Σ g_i·O_i:
    dL/da_i = g_i·(v1 − v0)·p_i(1 − p_i)·c·(k1 − k0); dL/dv1 = Σ g_i·p_i;
    dL/dv0 = Σ g_i·(1 − p_i); dL/dk1 = Σ g_i·(v1 − v0)·p_i(1 − p_i)·c·a_i = −dL/dk0."""
    a = np.array([0.8, -1.3])
    kk = np.array([0.4, 1.1])
    vv = np.array([2.0, -0.5])
    g = np.array([1.5, 0.25])
    c = 0.9
    q = a.reshape(1, 1, 2, 1)
    k = kk.reshape(1, 1, 2, 1)
    v = vv.reshape(1, 1, 2, 1)
    do = g.reshape(1, 1, 2, 1)
    dq, dk, dv = orc.attention_backward(q, k, v, do, False, c)
    p = 1.0 / (1.0 + np.exp(-c * a * (kk[1] - kk[0])))
    w = g * (vv[1] - vv[0]) * p * (1 - p) * c
    assert np.max(np.abs(dq[0, 0, :, 0] - w * (kk[1] - kk[0]))) <= 1e-14
    assert abs(dv[0, 0, 1, 0] - np.sum(g * p)) <= 1e-14
    assert abs(dv[0, 0, 0, 0] - np.sum(g * (1 - p))) <= 1e-14
    assert abs(dk[0, 0, 1, 0] - np.sum(w * a)) <= 1e-14
    assert abs(dk[0, 0, 0, 0] + np.sum(w * a)) <= 1e-14
    # causal: row 0 sees only key 0 (O_0 = v0); row 1 as above
    dq, dk, dv = orc.attention_backward(q, k, v, do, True, c)
    assert dq[0, 0, 0, 0] == 0.0
    assert abs(dq[0, 0, 1, 0] - w[1] * (kk[1] - kk[0])) <= 1e-14
    assert abs(dv[0, 0, 0, 0] - (g[0] + g[1] * (1 - p[1]))) <= 1e-14
    assert abs(dv[0, 0, 1, 0] - g[1] * p[1]) <= 1e-14
    assert abs(dk[0, 0, 1, 0] - w[1] * a[1]) <= 1e-14


def pin_bwd_invariants(orc):
    """Shifting every key by u leaves O unchanged, so Σ_j dK_j = 0; adding c to every
    value row adds c to every output row, so Σ_j dV_j = Σ_i dO_i; with V constant O does
    not depend on Q or K, so dQ = dK = 0; causal query 0 sees one key, so dQ_0 = 0, and
    the last key is seen by the last query alone: dV_{T−1} = P_{T−1,T−1}·dO_{T−1}."""
    B, H, T, d = 2, 2, 33, 5
    q, k, v = _qkv(21, B, H, T, d, std=1.3)
    do = _rng(22).standard_normal((B, H, T, d))
    scale = 0.45
    for causal in (False, True):
        dq, dk, dv = orc.attention_backward(q, k, v, do, causal, scale)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-12
        assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) <= 1e-12
        vc = np.broadcast_to(np.linspace(-1.0, 2.0, d), v.shape).copy()
        dq0, dk0, _ = orc.attention_backward(q, k, vc, do, causal, scale)
        assert np.max(np.abs(dq0)) <= 1e-12 and np.max(np.abs(dk0)) <= 1e-12
        if causal:
            assert np.max(np.abs(dq[:, :, 0])) == 0.0
            o, lse = orc.attention(q, k, v, True, scale)
            s_last = scale * np.einsum("bhd,bhd->bh", q[:, :, -1], k[:, :, -1])
            p_last = np.exp(s_last - lse[:, :, -1])
            assert np.max(np.abs(dv[:, :, -1] - p_last[..., None] * do[:, :, -1])) <= 1e-13


def pin_bwd_autograd(orc):
    """Cross-check against PyTorch autograd through its CPU scaled_dot_product_attention
    in fp64 (a library routine for the same derivative)."""
    import torch
    import torch.nn.functional as F
    q, k, v = _qkv(23, 2, 2, 41, 16)
    do = _rng(24).standard_normal(q.shape)
    for causal in (False, True):
        tq, tk, tv = (torch.from_numpy(t.copy()).requires_grad_(True) for t in (q, k, v))
        out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.25)
        out.backward(torch.from_numpy(do))
        got = orc.attention_backward(q, k, v, do, causal, 0.25)
        for g, t in zip(got, (tq, tk, tv)):
            assert np.max(np.abs(g - t.grad.numpy())) <= 1e-12


def pin_bwd_sampled(orc):
    """dQ of sampled query rows and dK, dV of sampled key rows equal the full gradient on
    those rows (several row chunks, a ragged last chunk)."""
    q, k, v = _qkv(25, 1, 1, 1100, 8)
    do = _rng(26).standard_normal(q.shape)
    rows = np.array([0, 1, 511, 512, 513, 1023, 1099])
    for causal in (False, True):
        dq, dk, dv = orc.attention_backward(q, k, v, do, causal, 0.3)
        dqr = orc.attention_backward_rows(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, 0.3, rows)
        dkc, dvc = orc.attention_backward_cols(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, 0.3,
                                               rows)
        assert np.max(np.abs(dqr - dq[0, 0, rows])) <= 1e-12
        assert np.max(np.abs(dkc - dk[0, 0, rows])) <= 1e-12
        assert np.max(np.abs(dvc - dv[0, 0, rows])) <= 1e-12


def pin_bwd_magnitudes(orc):
    """The error-bound magnitudes dominate the gradients (|Σ a·b| ≤ Σ|a|·|b|), and with
    dO ≥ 0 the dV magnitude is dV itself (P ≥ 0, so no term changes sign)."""
    q, k, v = _qkv(27, 1, 2, 70, 6)
    do = _rng(28).standard_normal(q.shape)
    for causal in (False, True):
        g = orc.attention_backward(q, k, v, do, causal, 0.4)
        m = orc.attention_backward_magnitudes(q, k, v, do, causal, 0.4)
        for gi, mi in zip(g, m):
            assert np.all(mi >= np.abs(gi) - 1e-12)
        dop = np.abs(do)
        _, _, dv = orc.attention_backward(q, k, v, dop, causal, 0.4)
        _, _, mv = orc.attention_backward_magnitudes(q, k, v, dop, causal, 0.4)
        assert np.max(np.abs(mv - dv)) <= 1e-12


# ------------------------------------------------------------- general form (Tq ≠ Tk, masks)

def brute_force_general(q, k, v, causal, scale, block_mask, block):
    """Pure-Python loops: query i sees key j iff (not causal or j ≤ i + Tk − Tq) and the
    block (i // block, j // block) is on; a row that sees nothing gives O = 0, LSE = −∞."""
    q = np.asarray(q).tolist()
    k = np.asarray(k).tolist()
    v = np.asarray(v).tolist()
    Tq, Tk, d = len(q), len(k), len(q[0])
    o = [[0.0] * d for _ in range(Tq)]
    lse = [-math.inf] * Tq
    for i in range(Tq):
        keys = [j for j in range(Tk)
                if (not causal or j <= i + Tk - Tq)
                and (block_mask is None or block_mask[i // block][j // block])]
        if not keys:
            continue
        s = {j: scale * sum(q[i][t] * k[j][t] for t in range(d)) for j in keys}
        m = max(s.values())
        e = {j: math.exp(s[j] - m) for j in keys}
        l = sum(e.values())
        for t in range(d):
            o[i][t] = sum(e[j] * v[j][t] for j in keys) / l
        lse[i] = m + math.log(l)
    return np.array(o), np.array(lse)


def pin_general_bruteforce(orc):
    """Tq ≠ Tk, bottom-right causal, random block masks (block = 2 rows/keys) including
    empty block rows: numpy general form == pure-Python loops within 1e-12."""
    r = _rng(40)
    for n, (Tq, Tk, causal) in enumerate([(3, 7, True), (5, 5, True), (4, 9, False), (1, 6, True),
                                          (7, 3, False), (6, 6, False)]):
        q = r.standard_normal((Tq, 3))
        k = r.standard_normal((Tk, 3))
        v = r.standard_normal((Tk, 3))
        for trial in range(3):
            bm = None if trial == 0 else (r.random(((Tq + 1) // 2, (Tk + 1) // 2)) < 0.6)
            if trial == 2:
                bm[0, :] = False   # an empty row block
            o, lse = orc.attention_general_head(q, k, v, causal, 0.8, bm, block=2)
            ob, lb = brute_force_general(q, k, v, causal, 0.8, bm, 2)
            assert np.max(np.abs(o - ob)) <= 1e-12, (n, trial)
            fin = np.isfinite(lb)
            assert np.array_equal(np.isneginf(lse), np.isneginf(lb)), (n, trial)
            assert np.all(np.abs(lse[fin] - lb[fin]) <= 1e-12), (n, trial)


def pin_general_reduces_to_attention(orc):
    """Tq = Tk with no block mask (or an all-ones one) is plain attention; a block mask
    that keeps exactly the blocks on or below the diagonal changes nothing under causal."""
    q, k, v = _qkv(41, 1, 2, 300, 8)
    for causal in (False, True):
        o, lse = orc.attention(q, k, v, causal, 0.3)
        og, lg = orc.attention_general(q, k, v, causal, 0.3)
        assert np.max(np.abs(o - og)) <= 1e-13 and np.max(np.abs(lse - lg)) <= 1e-13
        ones = np.ones((3, 3), dtype=np.uint8)
        og, lg = orc.attention_general(q, k, v, causal, 0.3, ones)
        assert np.max(np.abs(o - og)) <= 1e-13 and np.max(np.abs(lse - lg)) <= 1e-13
    tri = np.tril(np.ones((3, 3), dtype=np.uint8))
    o, lse = orc.attention(q, k, v, True, 0.3)
    og, lg = orc.attention_general(q, k, v, True, 0.3, tri)
    assert np.max(np.abs(o - og)) <= 1e-13 and np.max(np.abs(lse - lg)) <= 1e-13


def pin_general_decode(orc):
    """One query against Tk keys under causal (bottom-right) sees every key: it equals the
    last row of full causal attention over the same keys, and with q = 0 the mean of V with
    LSE = ln Tk. The causal rows of Tq < Tk equal the last Tq rows of full causal attention."""
    _, k, v = _qkv(42, 1, 1, 37, 5)
    q = _rng(43).standard_normal((1, 1, 1, 5))
    full_q = np.concatenate([_rng(44).standard_normal((1, 1, 36, 5)), q], axis=2)
    o_full, l_full = orc.attention(full_q, k, v, True, 0.6)
    o, lse = orc.attention_general(q, k, v, True, 0.6)
    assert np.max(np.abs(o[0, 0, 0] - o_full[0, 0, -1])) <= 1e-13
    assert abs(lse[0, 0, 0] - l_full[0, 0, -1]) <= 1e-13
    o, lse = orc.attention_general(np.zeros((1, 1, 1, 5)), k, v, True, 0.6)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 0].mean(axis=0))) <= 1e-13
    assert abs(lse[0, 0, 0] - math.log(37)) <= 1e-13
    o, lse = orc.attention_general(full_q[:, :, -9:], k, v, True, 0.6)
    assert np.max(np.abs(o - o_full[:, :, -9:])) <= 1e-13
    assert np.max(np.abs(lse - l_full[:, :, -9:])) <= 1e-13


def pin_general_empty_rows(orc):
    """A row block switched off entirely gives O = 0 and LSE = −∞ on exactly its rows."""
    q, k, v = _qkv(45, 1, 1, 40, 4)
    bm = np.ones((5, 5), dtype=np.uint8)
    bm[2, :] = 0
    o, lse = orc.attention_general(q, k, v, False, 0.5, bm, block=8)
    assert np.all(o[0, 0, 16:24] == 0.0) and np.all(np.isneginf(lse[0, 0, 16:24]))
    assert np.all(np.isfinite(lse[0, 0, :16])) and np.all(np.isfinite(lse[0, 0, 24:]))


def pin_merge_partials(orc):
    """Merging results over disjoint key ranges gives the full result: worked by hand for
    two parts (O = 1, LSE = ln 1 and O = 2, LSE = ln 3 → O = 7/4, LSE = ln 4), and on data
    with the key range split into 3 block ranges by block masks, causal and not, with one
    range that some rows never see (LSE = −∞, weight 0)."""
    o, lse = orc.merge_partials(np.array([[1.0], [2.0]]), np.array([0.0, math.log(3.0)]))
    assert abs(o[0] - 1.75) <= 1e-15 and abs(lse - math.log(4.0)) <= 1e-15
    q, k, v = _qkv(46, 1, 2, 24, 4)
    for causal in (False, True):
        o_full, l_full = orc.attention_general(q, k, v, causal, 0.7, None, block=8)
        parts_o, parts_l = [], []
        for s in range(3):
            bm = np.zeros((3, 3), dtype=np.uint8)
            bm[:, s] = 1
            po, pl = orc.attention_general(q, k, v, causal, 0.7, bm, block=8)
            parts_o.append(po)
            parts_l.append(pl)
        o, lse = orc.merge_partials(np.stack(parts_o), np.stack(parts_l))
        assert np.max(np.abs(o - o_full)) <= 1e-13 and np.max(np.abs(lse - l_full)) <= 1e-13
    # huge LSEs: the max shift keeps the merge finite
    o, lse = orc.merge_partials(np.array([[1.0], [3.0]]), np.array([900.0, 900.0]))
    assert abs(o[0] - 2.0) <= 1e-15 and abs(lse - (900.0 + math.log(2.0))) <= 1e-12


ORACLE_PINS = [pin_bruteforce, pin_hand_example, pin_row_sums, pin_constant_v,
               pin_causal_row0, pin_uniform, pin_shift, pin_permutation, pin_large_scores,
               pin_rows_match_full, pin_sdpa_library]
RECURRENCE_PINS = [pin_online_trace, pin_online_weighted_sum]
GENERAL_PINS = [pin_general_bruteforce, pin_general_reduces_to_attention, pin_general_decode,
                pin_general_empty_rows, pin_merge_partials]
BACKWARD_PINS = [pin_bwd_finite_diff, pin_bwd_hand_example, pin_bwd_invariants,
                 pin_bwd_autograd, pin_bwd_sampled, pin_bwd_magnitudes]


def load_page_facts():
    with open(os.path.join(GOLDEN, "page_facts.json"), encoding="utf-8") as f:
        return json.load(f)


def run_all(orc, pins):
    """Run pins; return the names of the ones that failed."""
    failed = []
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except (AssertionError, FloatingPointError, ValueError, IndexError) as e:  # noqa: F841
            failed.append(pin.__name__)
    return failed


__all__ = ["ORACLE_PINS", "RECURRENCE_PINS", "BACKWARD_PINS", "GENERAL_PINS", "run_all", "brute_force", "load_page_facts"]
