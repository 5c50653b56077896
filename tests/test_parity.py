"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle on the same
seeded bf16 inputs. Tolerances: O max-abs ≤ 2e-2 and mean-abs ≤ 1e-3; LSE ≤ 1e-3 absolute.

The bf16 rounding of the probabilities before the P·V product and of O at the end gives
errors of a few 1e-3 on O at these value scales; the fp32 running sum keeps LSE within
~1e-5. The bounds above leave room for that and nothing more."""

import math

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _torch():
    import torch
    return torch


def _run(q, k, v, causal, scale=None):
    import exact_attention_23_gb300 as fa
    torch = _torch()
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def _compare(o, lse, o_ref, lse_ref, what, rounding_allowance=False):
    """rounding_allowance: for edge shapes outside the named workloads (a handful of keys
    per row, so |O| ~ 1), add to the mean-abs bound the mean error that rounding O_ref to
    bf16 alone would make, 2^-9·mean|O_ref| (round-to-nearest costs between 2^-10 and
    2^-9 of a value on average). The named workloads use the plain bounds."""
    err = np.abs(o - o_ref)
    lerr = np.abs(lse - lse_ref)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    mean_bound = O_MEAN + (2.0 ** -9 * float(np.abs(o_ref).mean()) if rounding_allowance else 0.0)
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= mean_bound, f"{what}: O mean-abs {err.mean():.3e} > {mean_bound:.3e}"
    assert lerr.max() <= LSE_MAX, f"{what}: LSE max-abs {lerr.max():.3e}"
    return err.max(), err.mean(), lerr.max()


def _full_check(w, rounding_allowance=False):
    q, k, v = inputs.workload_qkv(w)
    o, lse = _run(q, k, v, w.causal)
    o_ref, lse_ref = oracle.attention(inputs.to_f64_numpy(q), inputs.to_f64_numpy(k),
                                      inputs.to_f64_numpy(v), w.causal, w.scale)
    return _compare(o, lse, o_ref, lse_ref, w.name, rounding_allowance)


@pytest.mark.parametrize("name,causal", [
    ("tiny_causal", True),
    ("ragged_t1000", True),
    ("ragged_t1000", False),
    ("gpt2_layer_spiky", True),
    ("gpt2_layer_spiky_q", True),
])
def test_parity_full(name, causal):
    _full_check(inputs.WORKLOADS[name].with_causal(causal))


@pytest.mark.parametrize("T", [1, 2, 100, 127, 128, 129, 255, 256, 257, 383, 384, 385, 640, 777])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_parity_ragged_lengths(T, d, causal):
    """Edge lengths: one row, a partial first tile, exact tiles, one past a tile, a lone
    last Q tile in a pair, and odd lengths."""
    w = inputs.Workload(f"edge_t{T}_d{d}", 1, 3, T, d, causal, 1000 + T + d)
    _full_check(w, rounding_allowance=True)


@pytest.mark.parametrize("T", [1100, 1281])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_parity_odd_tile_count_in_pairs(T, d, causal):
    """An odd number of 128-row query tiles while the kernel runs two tiles per work unit:
    the last unit of every head holds one tile, the producer still issues the pair's
    second (wholly out-of-range) query box and one softmax warpgroup sits that unit out.
    B4 H12 gives enough units that the host picks pairs (pairs at least fill the SMs)."""
    torch = _torch()
    B, H = 4, 12
    n_qt = -(-T // 128)
    assert n_qt % 2 == 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((n_qt + 1) // 2) * B * H >= sms, "the host would pick single-tile units"
    w = inputs.Workload(f"odd_tiles_t{T}_d{d}", B, H, T, d, causal, 2000 + T + d)
    _full_check(w)


@pytest.mark.parametrize("T", [1153, 1409])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_parity_ragged_in_pairs(T, d, causal):
    """Ragged last tiles (T not a multiple of 128) on the two-tile-per-CTA kernel: B4 H12 has
    enough pairs to fill the SMs, so the host runs pairs rather than single tiles."""
    torch = _torch()
    B, H = 4, 12
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert ((-(-T // 128) + 1) // 2) * B * H >= sms, "the host would pick single-tile units"
    _full_check(inputs.Workload(f"pairs_t{T}_d{d}", B, H, T, d, causal, 2500 + T + d))


@pytest.mark.parametrize("scale", [-0.125, -0.05])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_parity_negative_scale(scale, d, causal):
    """A negative factor on QKᵀ (the step S = QKᵀ/√d takes the factor from the caller): the
    row maximum of the scaled scores comes from the smallest raw score, and masked scores
    must still weigh nothing. Ragged T = 777 (a partial last tile)."""
    q, k, v = inputs.make_qkv(1, 3, 777, d, seed=3000 + d)
    o, lse = _run(q, k, v, causal, scale=scale)
    o_ref, lse_ref = oracle.attention(inputs.to_f64_numpy(q), inputs.to_f64_numpy(k),
                                      inputs.to_f64_numpy(v), causal, scale)
    _compare(o, lse, o_ref, lse_ref, f"scale {scale} d{d} causal={causal}",
             rounding_allowance=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_scale_zero_is_uniform_attention(d, causal):
    """scale = 0: every visible key weighs the same, whatever q and k hold. O_i is the mean
    of the visible v rows and LSE_i = ln(visible count): the closed form, and the oracle
    agrees. T = 333 (ragged)."""
    T = 333
    q, k, v = inputs.make_qkv(1, 2, T, d, seed=3100 + d)
    o, lse = _run(q, k, v, causal, scale=0.0)
    vv = inputs.to_f64_numpy(v)
    if causal:
        want_o = np.cumsum(vv, axis=2) / np.arange(1, T + 1)[None, None, :, None]
        want_l = np.log(np.arange(1, T + 1))[None, None]
    else:
        want_o = np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
        want_l = np.full((1, 2, T), math.log(T))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.max(np.abs(o - want_o)) <= O_MAX
    assert np.max(np.abs(lse - want_l)) <= LSE_MAX
    o_ref, lse_ref = oracle.attention(inputs.to_f64_numpy(q), inputs.to_f64_numpy(k), vv, causal,
                                      0.0)
    _compare(o, lse, o_ref, lse_ref, f"scale 0 d{d} causal={causal}", rounding_allowance=True)


def _sample_rows(T, rng, n_random=48):
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, T // 2, T - 129, T - 128, T - 2, T - 1]
    rows = set(r for r in fixed if 0 <= r < T)
    rows.update(int(x) for x in rng.integers(0, T, n_random))
    return np.array(sorted(rows))


def _sampled_check(w, bh_samples=3):
    torch = _torch()
    import exact_attention_23_gb300 as fa
    q, k, v = inputs.workload_qkv(w)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed + 77)
    BH = w.B * w.H
    worst = (0.0, 0.0, 0.0)
    for bh in sorted(set([0, BH - 1] + [int(x) for x in rng.integers(0, BH, bh_samples)])):
        b, h = divmod(bh, w.H)
        rows = _sample_rows(w.T, rng)
        o_ref, lse_ref = oracle.attention_rows(
            inputs.to_f64_numpy(q[b, h]), inputs.to_f64_numpy(k[b, h]),
            inputs.to_f64_numpy(v[b, h]), w.causal, w.scale, rows)
        og = o[b, h][torch.from_numpy(rows).cuda()].float().cpu().double().numpy()
        lg = lse[b, h][torch.from_numpy(rows).cuda()].cpu().double().numpy()
        r = _compare(og, lg, o_ref, lse_ref, f"{w.name} bh={bh}")
        worst = tuple(max(a, c) for a, c in zip(worst, r))
    # properties that hold at any size
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())
    if w.causal:
        assert torch.equal(o[:, :, 0], vd[:, :, 0]), "causal row 0 must equal v0 bit for bit"
    return worst


@pytest.mark.parametrize("T", inputs.SWEEP_T)
def test_parity_sweep_sampled(T):
    _sampled_check(inputs.WORKLOADS[f"sweep_t{T}"])


@pytest.mark.parametrize("causal", [True, False])
def test_parity_wide_head_t16k_sampled(causal):
    _sampled_check(inputs.WORKLOADS["wide_head_t16k"].with_causal(causal))


@pytest.mark.parametrize("name,causal", [
    ("sweep_t16384", True),
    ("wide_head_t16k", True),
    ("wide_head_t16k", False),
])
def test_parity_whole_heads_t16k(name, causal):
    """Every row of two whole heads (the first and the last (batch, head) of the launch) at
    the full 16384-row size, against the oracle's full attention of those heads: each
    tile position, both ends of the zig-zag unit order and every K step of the last
    tiles, under the same element-wise tolerances as the small workloads."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    w = inputs.WORKLOADS[name].with_causal(causal)
    q, k, v = inputs.workload_qkv(w)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=w.causal)
    torch.cuda.synchronize()
    for bh in (0, w.B * w.H - 1):
        b, h = divmod(bh, w.H)
        o_ref, lse_ref = oracle.attention(
            *(inputs.to_f64_numpy(t[b:b + 1, h:h + 1]) for t in (q, k, v)), w.causal, w.scale)
        og = o[b:b + 1, h:h + 1].float().cpu().double().numpy()
        lg = lse[b:b + 1, h:h + 1].cpu().double().numpy()
        _compare(og, lg, o_ref, lse_ref, f"{w.name} causal={causal} bh={bh} (all rows)")


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row0_bit_exact_and_lse(d):
    torch = _torch()
    q, k, v = inputs.make_qkv(2, 3, 300, d, seed=41)
    o, lse = _run(q, k, v, True)
    assert np.array_equal(o[:, :, 0], inputs.to_f64_numpy(v[:, :, 0]))
    want = (1.0 / math.sqrt(d)) * np.einsum("bhd,bhd->bh", inputs.to_f64_numpy(q[:, :, 0]),
                                            inputs.to_f64_numpy(k[:, :, 0]))
    assert np.max(np.abs(lse[:, :, 0] - want)) <= LSE_MAX
    del torch


@pytest.mark.parametrize("d", [64, 128])
def test_uniform_attention_closed_form(d):
    """q = 0: O_i is the mean of the visible v rows and LSE_i = ln(visible count). Pins the
    LSE base and the causal/padding masks on the GPU without the oracle."""
    torch = _torch()
    T = 333
    _, k, v = inputs.make_qkv(1, 2, T, d, seed=42)
    q = torch.zeros_like(k)
    vv = inputs.to_f64_numpy(v)
    o, lse = _run(q, k, v, True)
    cum = np.cumsum(vv, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    assert np.max(np.abs(o - cum)) <= O_MAX
    assert np.max(np.abs(lse - np.log(np.arange(1, T + 1))[None, None])) <= LSE_MAX
    o, lse = _run(q, k, v, False)
    assert np.max(np.abs(o - vv.mean(axis=2, keepdims=True))) <= O_MAX
    assert np.max(np.abs(lse - math.log(T))) <= LSE_MAX


def test_constant_v():
    torch = _torch()
    q, k, _ = inputs.make_qkv(1, 4, 700, 64, seed=43, std=2.0)
    c = torch.linspace(-2.0, 3.0, 64).to(torch.bfloat16)
    v = c.expand(1, 4, 700, 64).contiguous()
    for causal in (True, False):
        o, _ = _run(q, k, v, causal)
        assert np.max(np.abs(o - c.double().numpy())) <= O_MAX


def test_deterministic():
    torch = _torch()
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(2, 4, 1500, 64, seed=44))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_timeout_path_reports_status_and_context_survives():
    """A wait that can never complete (the query-tile loads are withheld) must give up,
    report FA_ERR_TIMEOUT through the status word and write NaN, leaving the context
    usable for the next call."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(1, 2, 512, 64, seed=45))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=True, status=status, timeout_ns=20_000_000,
                    flags=fa.FA_FLAG_TEST_STARVE_Q)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.FA_ERR_TIMEOUT
    assert bool(torch.isnan(lse).all()) and bool(torch.isnan(o.float()).all())
    status.zero_()
    o, lse = fa.fwd(q, k, v, causal=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, lse_ref = oracle.attention(*(inputs.to_f64_numpy(t.cpu()) for t in (q, k, v)), True,
                                      0.125)
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             "after timeout")


def test_timeout_after_a_finished_unit_reports_status_and_context_survives():
    """Each CTA's first work unit gets its query tiles, later units do not: the first unit
    completes and its epilogue waits (deferred into the next unit's first step) when the
    next unit's waits run out. The kernel must report FA_ERR_TIMEOUT, write NaN for every
    row it owns (the finished unit's included: its epilogue is abandoned with the rest),
    and leave the context usable. B4 H12 T4096 gives every CTA at least five units."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    q, k, v = (t.cuda() for t in inputs.make_qkv(4, 12, 4096, 64, seed=46))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=True, status=status, timeout_ns=20_000_000,
                    flags=fa.FA_FLAG_TEST_STARVE_LATER_Q)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.FA_ERR_TIMEOUT
    assert bool(torch.isnan(lse).all()) and bool(torch.isnan(o.float()).all())
    status.zero_()
    o, lse = fa.fwd(q, k, v, causal=True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = np.array([0, 1, 127, 128, 2047, 4095])
    qn, kn, vn = (inputs.to_f64_numpy(t[1, 7].cpu()) for t in (q, k, v))
    o_ref, lse_ref = oracle.attention_rows(qn, kn, vn, True, 0.125, rows)
    _compare(o[1, 7, rows].float().cpu().double().numpy(), lse[1, 7, rows].cpu().double().numpy(),
             o_ref, lse_ref, "after timeout")


def test_misaligned_pointer_rejected_on_device():
    torch = _torch()
    import exact_attention_23_gb300 as fa
    buf = torch.zeros(4 * 128 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    q = buf[1:1 + 128 * 64]  # 2-byte offset
    rc = fa.fa_fwd(q.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                   buf.data_ptr(), 1, 1, 128, 64, 1, 0.125, None)
    assert rc == fa.FA_ERR_MISALIGNED
