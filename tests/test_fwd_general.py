"""GPU parity of the general forward forms against the fp64 oracle's general form:
fa_fwd_kv (Tq queries over Tk keys, bottom-right causal, key range split over CTAs with
the partial results merged; Tq ≤ 2 runs the CUDA-core decode kernels) and
fa_fwd_block_sparse (128×128 blocks switched off).

Tolerances as for the forward: O max-abs ≤ 2e-2, mean-abs ≤ 1e-3 (+ 2⁻⁹·mean|O_ref| for
shapes whose rows see few keys, as in test_parity.py), LSE ≤ 1e-3 absolute on rows that see
a key. Rows that see no key must be exactly O = 0 and LSE = −∞. Inputs: q, k, v drawn by
inputs.make_qkv at the key length; the queries are the last Tq rows of that q draw (new
tokens at the end of the sequence)."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _compare(o, lse, o_ref, lse_ref, what):
    live = np.isfinite(lse_ref)
    assert np.all(np.isfinite(o)), what
    assert np.array_equal(np.isneginf(lse), ~live), f"{what}: empty rows differ"
    assert np.all(o[~live] == 0.0), f"{what}: empty rows must be 0"
    err = np.abs(o - o_ref)
    mean_bound = O_MEAN + 2.0 ** -9 * float(np.abs(o_ref).mean())
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= mean_bound, f"{what}: O mean-abs {err.mean():.3e} > {mean_bound:.3e}"
    if live.any():
        lerr = np.abs(lse[live] - lse_ref[live])
        assert lerr.max() <= LSE_MAX, f"{what}: LSE max-abs {lerr.max():.3e}"


def _qkv_kv(B, H, Tq, Tk, d, seed):
    q, k, v = inputs.make_qkv(B, H, Tk, d, seed)
    return q[:, :, Tk - Tq:].contiguous() if Tq <= Tk else inputs.make_qkv(B, H, Tq, d, seed)[0], k, v


@pytest.mark.parametrize("B,H,Tq,Tk,d,causal,n_splits", [
    (2, 12, 1, 4096, 64, True, 0),     # decode, automatic ranges
    (2, 12, 1, 4096, 64, True, 1),     # decode, one range
    (2, 12, 1, 4096, 64, True, 5),     # uneven ranges
    (1, 3, 1, 1, 64, True, 0),         # decode against a single cached key
    (1, 3, 1, 5, 128, True, 8),        # more ranges requested than keys
    (2, 6, 1, 8192, 128, False, 3),
    (1, 4, 1, 777, 64, True, 0),       # ragged cache length
    (1, 8, 1, 1000, 128, False, 0),
    (2, 4, 7, 2000, 64, True, 3),
    # two query rows (the CUDA-core multi-query decode): single and split key ranges, a tiny
    # cache; then the first tensor-core sizes
    (2, 12, 2, 4096, 64, True, 0),
    (1, 4, 2, 3000, 128, False, 5),
    (1, 4, 2, 5, 64, True, 0),         # fewer cached keys than a chunk
    (1, 4, 3, 5, 64, True, 0),         # fewer cached keys than a chunk
    (2, 6, 4, 3000, 128, True, 1),
    (1, 3, 4, 4, 64, True, 3),         # Tq = Tk = 4: plain causal attention, more ranges than keys allow
    (1, 4, 5, 777, 64, False, 0),
    (2, 3, 8, 8192, 64, True, 0),
    (1, 3, 9, 9, 128, True, 0),
    (2, 4, 16, 2500, 64, True, 7),
    (1, 4, 128, 1024, 64, True, 0),
    (1, 4, 200, 1500, 128, True, 0),   # two query tiles, ragged
    (1, 2, 300, 300, 64, True, 0),     # Tq = Tk: plain causal attention
    (1, 2, 1000, 300, 64, False, 2),   # more queries than keys (non-causal)
])
def test_fwd_kv_parity(B, H, Tq, Tk, d, causal, n_splits):
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = _qkv_kv(B, H, Tq, Tk, d, 500 + Tq + Tk + d)
    o, lse = fa.fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=causal, n_splits=n_splits)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_general(*(inputs.to_f64_numpy(t) for t in (q, k, v)),
                                              causal, d ** -0.5)
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             f"kv B{B} H{H} Tq{Tq} Tk{Tk} d{d} causal={causal} splits={n_splits}")


def test_fwd_kv_equal_lengths_matches_fwd():
    """With Tq = Tk, no split and no mask the general form computes plain attention."""
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 6, 777, 64, 61))
    for causal in (True, False):
        o1, l1 = fa.fwd(q, k, v, causal=causal)
        o2, l2 = fa.fwd_kv(q, k, v, causal=causal, n_splits=1)
        torch.cuda.synchronize()
        assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
        assert (l1 - l2).abs().max().item() <= 1e-3


def _mask(nb, heads, density, seed, empty_row=None):
    r = np.random.default_rng(seed)
    m = (r.random((heads, nb, nb)) < density).astype(np.uint8)
    if empty_row is not None:
        m[:, empty_row, :] = 0
    return m


@pytest.mark.parametrize("T,d,causal,per_head", [
    (256, 64, False, False),
    (1000, 64, True, False),
    (1000, 128, False, True),
    (2048, 64, True, True),
    (777, 128, True, False),
])
def test_fwd_block_sparse_parity(T, d, causal, per_head):
    import torch
    import exact_attention_23_gb300 as fa
    B, H = 2, 3
    nb = fa.q_tiles(T)
    q, k, v = inputs.make_qkv(B, H, T, d, 700 + T + d)
    heads = B * H if per_head else 1
    m = _mask(nb, heads, 0.5, T + d, empty_row=1 if nb > 1 else None)
    mt = torch.from_numpy(m if per_head else m[0]).cuda().contiguous()
    o, lse = fa.fwd_block_sparse(q.cuda(), k.cuda(), v.cuda(), mt, causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_general(*(inputs.to_f64_numpy(t) for t in (q, k, v)),
                                              causal, d ** -0.5, m if per_head else m[0])
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             f"block-sparse T{T} d{d} causal={causal} per_head={per_head}")


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_fwd_block_sparse_many_units_per_cta(d, causal):
    """B4 H12 T4096: 768 units, five or more per CTA, so each softmax warpgroup ends units
    and starts new ones inside one launch (at d = 64 the epilogue of each is deferred into
    the next). Per-head masks at half density, with a different empty block row in every
    head: some units then hold a Q tile that uses no K tile at all. Heads whose CTAs differ
    are checked in full against the oracle."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T = 4, 12, 4096
    nb = fa.q_tiles(T)
    q, k, v = inputs.make_qkv(B, H, T, d, 740 + d)
    m = _mask(nb, B * H, 0.5, 741 + d)
    for hh in range(B * H):
        m[hh, (3 * hh) % nb, :] = 0
    o, lse = fa.fwd_block_sparse(q.cuda(), k.cuda(), v.cuda(),
                                 torch.from_numpy(m).cuda().contiguous(), causal=causal)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for b, h in ((0, 0), (1, 5), (3, 11)):
        o_ref, lse_ref = oracle.attention_general_head(
            *(inputs.to_f64_numpy(t[b, h]) for t in (q, k, v)), causal, d ** -0.5, m[b * H + h])
        _compare(o[b, h], lse[b, h], o_ref, lse_ref,
                 f"block-sparse many units d{d} causal={causal} head ({b},{h})")


def test_fwd_kv_prefill_many_units_per_cta_d128():
    """B2 H12, 2048 new queries against 4096 cached keys at d = 128, bottom-right causal,
    one key range: 192 units over the SMs, so CTAs run several in turn (P in two halves,
    output through the staging slices). Rows sampled in three heads."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, Tq, Tk, d = 2, 12, 2048, 4096, 128
    q, k, v = _qkv_kv(B, H, Tq, Tk, d, 750)
    o, lse = fa.fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=True, n_splits=1)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    rows = np.array([0, 1, 127, 128, 1023, 1024, 2047])
    for b, h in ((0, 0), (1, 6), (1, 11)):
        qn, kn, vn = (inputs.to_f64_numpy(t[b, h]) for t in (q, k, v))
        # new query r is token Tk − Tq + r: it sees the keys up to and including that one
        for r in rows:
            o1, l1 = oracle.attention_general(qn[r:r + 1][None, None],
                                              kn[:Tk - Tq + r + 1][None, None],
                                              vn[:Tk - Tq + r + 1][None, None], False, d ** -0.5)
            _compare(o[b, h, r:r + 1], lse[b, h, r:r + 1], o1[0, 0], l1[0, 0],
                     f"kv prefill d128 head ({b},{h}) row {r}")


@pytest.mark.parametrize("d,causal", [(64, True), (128, False)])
def test_fwd_kv_pairs_with_split_ranges(d, causal):
    """B4 H12, 512 new queries against 16384 cached keys, automatic ranges: on a 152-SM GB300
    the cost rule picks 3 key ranges, and the 48 · 2 · 3 = 288 pair units fill the SMs, so the
    pair kernel's general form runs with split ranges (fp32 partial rows, then the merge).
    Every row of three heads against the oracle."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, Tq, Tk = 4, 12, 512, 16384
    assert fa.fa_fwd_kv_workspace_size(B, H, Tq, Tk, d, 0) > 0, "expected split key ranges"
    q, k, v = _qkv_kv(B, H, Tq, Tk, d, 760 + d)
    o, lse = fa.fwd_kv(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for b, h in ((0, 0), (2, 7), (3, 11)):
        o_ref, lse_ref = oracle.attention_general_head(
            *(inputs.to_f64_numpy(t[b, h]) for t in (q, k, v)), causal, d ** -0.5)
        _compare(o[b, h], lse[b, h], o_ref, lse_ref,
                 f"kv pairs+ranges d{d} causal={causal} head ({b},{h})")


def test_fwd_block_sparse_full_and_causal_masks():
    """An all-ones mask is plain attention; keeping the blocks on and below the diagonal
    under causal is plain causal attention (the skipped blocks were fully masked)."""
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 4, 1000, 64, 71))
    nb = fa.q_tiles(1000)
    ones = torch.ones((nb, nb), dtype=torch.uint8, device="cuda")
    tril = torch.tril(ones).contiguous()
    o_ref, l_ref = fa.fwd(q, k, v, causal=False)
    o, l = fa.fwd_block_sparse(q, k, v, ones, causal=False)
    oc_ref, lc_ref = fa.fwd(q, k, v, causal=True)
    oc, lc = fa.fwd_block_sparse(q, k, v, tril, causal=True)
    torch.cuda.synchronize()
    assert (o.float() - o_ref.float()).abs().max().item() <= 2e-2
    assert (l - l_ref).abs().max().item() <= 1e-3
    assert (oc.float() - oc_ref.float()).abs().max().item() <= 2e-2
    assert (lc - lc_ref).abs().max().item() <= 1e-3


def test_fwd_block_sparse_all_off():
    """A mask with every block off: every row is empty (O = 0, LSE = −∞)."""
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 300, 64, 72))
    zeros = torch.zeros((3, 3), dtype=torch.uint8, device="cuda")
    o, lse = fa.fwd_block_sparse(q, k, v, zeros, causal=True)
    torch.cuda.synchronize()
    assert bool((o == 0).all()) and bool(torch.isneginf(lse).all())
