"""GPU parity of the backward pass: dQ, dK, dV from the CUDA path (forward kernel, then
backward kernel, both through the C ABI) against the fp64 CPU oracle's gradient on the
same seeded bf16 q, k, v, dO.

Tolerance, element by element (full-size comparisons), for a gradient G:

    |G − G_ref| ≤ 2^-8·|G_ref| + 2^-7·M_G + 1e-6

where M_G is the oracle's error-bound magnitude of that element's sum (the same sum with
every term in absolute value; see oracle.attention_backward_magnitudes). Derivation: the
kernel rounds P and dS to bf16 (unit roundoff u = 2^-8) before the tensor-core products
and builds D = Σ dO∘O from the bf16 O of the forward, so to first order each term of a
gradient sum carries a relative error ≤ u, and the sum is off by ≤ u·M_G; the final bf16
rounding of G adds ≤ u·|G|. The bound doubles the first term's constant; replaying the
kernel's roundings in fp64 on these workloads reaches at most 0.65 of u·M_G. The last term
covers fp32 noise where the exact gradient is 0 (causal query 0: dQ_0 = 0).

Whole heads of the full-size launches (T = 16384 at d = 64, T = 8192 at d = 128) are
checked element by element under that bound, the oracle computing the magnitudes of those
heads alone. Sampled checks across the other heads (T = 4096, 16384), where the magnitudes
of every head would cost a full backward on the CPU, use scale-relative bounds instead:
    max|G − G_ref| ≤ 2e-2·max|G_ref|,   mean|G − G_ref| ≤ 5e-3·mean|G_ref|
(the replay above gives at most 5.7e-3 and 2.3e-3 for these ratios at T ≥ 256). A dropped
term, a wrong mask or a transposed operand gives errors of order 1 under either bound."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

U = 2.0 ** -8                      # bf16 unit roundoff
REL_MAX, REL_MEAN = 2e-2, 5e-3     # sampled checks
ABS_FLOOR = 1e-6


def _torch():
    import torch
    return torch


def _run(q, k, v, do, causal, workspace=None):
    """Forward then backward on the GPU; returns (dq, dk, dv) as fp64 numpy arrays."""
    import exact_attention_23_gb300 as fa
    torch = _torch()
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, workspace=workspace)
    torch.cuda.synchronize()
    return tuple(t.float().cpu().double().numpy() for t in (dq, dk, dv))


def _compare_elementwise(got, ref, mags, what):
    worst = []
    for name, g, r, m in zip(("dQ", "dK", "dV"), got, ref, mags):
        assert np.all(np.isfinite(g)), f"{what}: {name} not finite"
        err = np.abs(g - r)
        bound = U * np.abs(r) + 2.0 * U * m + ABS_FLOOR
        ratio = err / bound
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        assert ratio[i] <= 1.0, (f"{what}: {name}{list(i)} err {err[i]:.3e} > bound "
                                 f"{bound[i]:.3e} (ref {r[i]:.3e}, magnitude {m[i]:.3e})")
        worst.append(float(ratio[i]))
    return worst


def _compare_relative(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(g)), f"{what}: {name} not finite"
        err = np.abs(g - r)
        smax, smean = float(np.abs(r).max()), float(np.abs(r).mean())
        assert err.max() <= REL_MAX * smax + ABS_FLOOR, \
            f"{what}: {name} max-abs {err.max():.3e} > {REL_MAX} × {smax:.3e}"
        assert err.mean() <= REL_MEAN * smean + ABS_FLOOR, \
            f"{what}: {name} mean-abs {err.mean():.3e} > {REL_MEAN} × {smean:.3e}"


def _full_check(w):
    q, k, v = inputs.workload_qkv(w)
    do = inputs.workload_do(w)
    got = _run(q, k, v, do, w.causal)
    args = [inputs.to_f64_numpy(t) for t in (q, k, v, do)]
    ref = oracle.attention_backward(*args, w.causal, w.scale)
    mags = oracle.attention_backward_magnitudes(*args, w.causal, w.scale)
    return _compare_elementwise(got, ref, mags, w.name)


@pytest.mark.parametrize("name,causal", [
    ("tiny_causal", True),
    ("tiny_causal", False),
    ("ragged_t1000", True),
    ("ragged_t1000", False),
    ("gpt2_layer_spiky", True),
    ("gpt2_layer_spiky_q", True),
])
def test_bwd_parity_full(name, causal):
    _full_check(inputs.WORKLOADS[name].with_causal(causal))


@pytest.mark.parametrize("T", [1, 2, 100, 127, 128, 129, 255, 256, 257, 385, 640, 777])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_parity_ragged_lengths(T, causal):
    """One row, a partial first tile, exact tiles, one past a tile, odd lengths."""
    _full_check(inputs.Workload(f"bwd_edge_t{T}", 1, 3, T, 64, causal, 2000 + T))


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 200, 256, 385, 777, 1024])
@pytest.mark.parametrize("causal", [True, False])
def test_bwd_parity_d128(T, causal):
    """Head dim 128 (64-query tiles, dQ made transposed): lengths around the 64-row query
    tiles and the 128-row key tiles."""
    _full_check(inputs.Workload(f"bwd_d128_t{T}", 2, 2, T, 128, causal, 3000 + T))


def _sample(T, rng, n_random=24):
    fixed = [0, 1, 127, 128, 129, T // 2, T - 129, T - 128, T - 2, T - 1]
    s = set(r for r in fixed if 0 <= r < T)
    s.update(int(x) for x in rng.integers(0, T, n_random))
    return np.array(sorted(s))


def _sampled_check(w, heads=2):
    """Full-size workload: dQ on sampled query rows, dK and dV on sampled key rows of a
    few heads, each computed by the oracle one row (or column of P) at a time."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    q, k, v = inputs.workload_qkv(w)
    do = inputs.workload_do(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=w.causal)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t.float()).all())
    rng = np.random.default_rng(w.seed + 99)
    BH = w.B * w.H
    for bh in sorted(set([0, BH - 1] + [int(x) for x in rng.integers(0, BH, heads)])):
        b, h = divmod(bh, w.H)
        rows = _sample(w.T, rng)
        args = [inputs.to_f64_numpy(t[b, h]) for t in (q, k, v, do)]
        dq_ref = oracle.attention_backward_rows(*args, w.causal, w.scale, rows)
        dk_ref, dv_ref = oracle.attention_backward_cols(*args, w.causal, w.scale, rows)
        idx = torch.from_numpy(rows).cuda()
        got = tuple(t[b, h][idx].float().cpu().double().numpy() for t in (dq, dk, dv))
        _compare_relative(got, (dq_ref, dk_ref, dv_ref), f"{w.name} bh={bh}")


@pytest.mark.parametrize("name,causal,bh", [
    ("sweep_t16384", True, 47),
    ("bwd_d128_t8192", False, 0),
])
def test_bwd_parity_whole_head_full_size(name, causal, bh):
    """One whole head of a full-size launch (every row of dQ, dK and dV) under the
    element-wise bound of the small workloads, with the oracle's magnitudes for that head:
    the d = 64 causal sweep at T = 16384 (its last (batch, head)) and the d = 128
    non-causal T = 8192 workload (its first)."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    w = (inputs.WORKLOADS[name] if name in inputs.WORKLOADS
         else inputs.Workload(name, 2, 8, 8192, 128, causal, 32)).with_causal(causal)
    q, k, v = inputs.workload_qkv(w)
    do = inputs.workload_do(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=w.causal)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=w.causal)
    torch.cuda.synchronize()
    b, h = divmod(bh, w.H)
    got = tuple(t[b:b + 1, h:h + 1].float().cpu().double().numpy() for t in (dq, dk, dv))
    args = [inputs.to_f64_numpy(t[b:b + 1, h:h + 1]) for t in (q, k, v, do)]
    ref = oracle.attention_backward(*args, w.causal, w.scale)
    mags = oracle.attention_backward_magnitudes(*args, w.causal, w.scale)
    _compare_elementwise(got, ref, mags, f"{w.name} bh={bh} (whole head)")


@pytest.mark.parametrize("T", [4096, 16384])
def test_bwd_parity_sweep_sampled(T):
    _sampled_check(inputs.WORKLOADS[f"sweep_t{T}"])


def test_bwd_parity_non_causal_long_sampled():
    w = inputs.Workload("bwd_noncausal_t4096", 2, 4, 4096, 64, False, 31)
    _sampled_check(w)


@pytest.mark.parametrize("causal", [True, False])
def test_bwd_parity_d128_long_sampled(causal):
    _sampled_check(inputs.Workload("bwd_d128_t8192", 2, 8, 8192, 128, causal, 32))


def test_bwd_workspace_reuse_and_determinism():
    """The call re-initialises its workspace (a reused, dirty workspace gives the same
    answer); dK and dV involve no atomics and are bit-identical between runs, dQ is summed
    with atomic adds in an unspecified order and agrees within rounding."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    w = inputs.WORKLOADS["ragged_t1000"]
    q, k, v = inputs.workload_qkv(w)
    do = inputs.workload_do(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    ws = fa.bwd_workspace(w.B, w.H, w.T, w.d, device=qd.device)
    ws.fill_(0x7F)  # garbage: a NaN-like pattern in every fp32 slot
    a = fa.bwd(qd, kd, vd, o, lse, dod, causal=True, workspace=ws)
    a = tuple(t.clone() for t in a)
    b = fa.bwd(qd, kd, vd, o, lse, dod, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    diff = (a[0].float() - b[0].float()).abs().max().item()
    assert diff <= 2e-2 * a[0].float().abs().max().item()


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_timeout_reports_and_poisons(d):
    """A wait that runs out (the query loads are withheld on purpose) stores
    FA_ERR_TIMEOUT and leaves NaN gradients; the next normal call is correct. Head dim 128
    has its own warp roles (a separate dQ issuer), so both are run."""
    torch = _torch()
    import exact_attention_23_gb300 as fa
    w = inputs.WORKLOADS["tiny_causal"] if d == 64 else inputs.Workload("tiny_wide", 1, 2, 256, 128, True, 12)
    q, k, v = inputs.workload_qkv(w)
    do = inputs.workload_do(w)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=True, status=status,
                        timeout_ns=20_000_000, flags=fa.FA_FLAG_TEST_STARVE_Q)
    torch.cuda.synchronize()
    assert int(status.item()) == fa.FA_ERR_TIMEOUT
    for t in (dq, dk, dv):
        assert bool(torch.isnan(t.float()).all())
    _full_check(w)


def test_bwd_rejects_bad_workspace():
    torch = _torch()
    import exact_attention_23_gb300 as fa
    x = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 256, dtype=torch.float32, device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.bwd(x, x.clone(), x.clone(), x.clone(), lse, x.clone(), workspace=small)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    with pytest.raises(fa.FAError):
        y = torch.zeros(1, 2, 256, 96, dtype=torch.bfloat16, device="cuda")
        fa.bwd(y, y.clone(), y.clone(), y.clone(), lse, y.clone())
