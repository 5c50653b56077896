"""GPU parity on inputs built to stress the online softmax's lazy rescale: O and l keep a
stale reference max until a score exceeds it by τ = 8 (base 2), then both are rescaled.

* Rising max: every query is the all-ones vector and key j is c·j·(1, …, 1), so the score
  grows along the keys. Each 128-key tile raises the row max by about 10 in base 2, more
  than τ, so every tile past the first forces a rescale (for the forward kernel's tiles and
  the decode kernel's key groups alike).
* Large magnitudes: q and k scaled by 16, so scores reach thousands and each row's softmax
  is nearly one-hot.

The oracle (fp64, the plain definition) decides; tolerances are the forward's, with the
rounding allowance of the edge-shape tests, since |O| is of order 1 here."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _score_error_bound(q, k, scale):
    """Per query row, a bound on the fp32 rounding of scale·q·k over d products:
    2·d·2⁻²⁴·scale·max_j Σ_c |q_c·k_jc| (the standard dot-product bound, doubled)."""
    qa = np.abs(inputs.to_f64_numpy(q))
    ka = np.abs(inputs.to_f64_numpy(k))
    d = qa.shape[-1]
    return 2.0 * d * 2.0 ** -24 * scale * np.max(qa @ np.swapaxes(ka, -1, -2), axis=-1)


def _compare(o, lse, o_ref, lse_ref, what, ds=None, vmax=0.0):
    """ds: per-row bound on the score error (natural units). It adds to the LSE tolerance,
    and 2·ds·max|v| adds to the O tolerance (a weight moves by at most its score error, and
    O is a convex combination of the rows of v)."""
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    extra = 0.0 if ds is None else 2.0 * float(ds.max()) * vmax
    mean_bound = O_MEAN + 2.0 ** -9 * float(np.abs(o_ref).mean()) + extra
    assert err.max() <= O_MAX + extra, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= mean_bound, f"{what}: O mean-abs {err.mean():.3e}"
    lerr = np.abs(lse - lse_ref)
    tol = LSE_MAX + (0.0 if ds is None else ds)
    assert np.all(lerr <= tol), f"{what}: LSE max-abs {lerr.max():.3e}"


def _rising(B, H, T, d, seed):
    """q = 1, k_j = c·j·1 (c gives ≈ 10 base-2 units of score per 128 keys at scale 1/√d),
    v from the seeded draw; all bf16."""
    import torch
    _, _, v = inputs.make_qkv(B, H, T, d, seed)
    scale = d ** -0.5
    c = 10.0 / (1.4426950408889634 * scale * d * 128)
    j = torch.arange(T, dtype=torch.float32)
    k = (c * j)[None, None, :, None].expand(B, H, T, d).to(torch.bfloat16).contiguous()
    q = torch.ones((B, H, T, d), dtype=torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("T,d,causal", [(1024, 64, True), (1024, 64, False),
                                        (777, 128, True), (1000, 128, False)])
def test_forward_rising_max_rescales_every_tile(T, d, causal):
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = _rising(1, 2, T, d, 900 + T)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(*(inputs.to_f64_numpy(t) for t in (q, k, v)), causal,
                                      d ** -0.5)
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             f"rising T{T} d{d} causal={causal}")


@pytest.mark.parametrize("Tk,d", [(4096, 64), (3000, 128)])
def test_decode_rising_max(Tk, d):
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = _rising(2, 3, Tk, d, 910 + Tk)
    q1 = q[:, :, -1:].contiguous()
    o, lse = fa.fwd_kv(q1.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_general(*(inputs.to_f64_numpy(t) for t in (q1, k, v)),
                                              True, d ** -0.5)
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             f"decode rising Tk{Tk} d{d}")


@pytest.mark.parametrize("d,causal", [(64, True), (128, False)])
def test_large_magnitude_scores(d, causal):
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = inputs.make_qkv(1, 3, 1000, d, 920 + d)
    q = (q.float() * 16).to(torch.bfloat16)
    k = (k.float() * 16).to(torch.bfloat16)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(*(inputs.to_f64_numpy(t) for t in (q, k, v)), causal,
                                      d ** -0.5)
    ds = _score_error_bound(q, k, d ** -0.5)
    vmax = float(np.abs(inputs.to_f64_numpy(v)).max())
    _compare(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
             f"large d{d} causal={causal}", ds=ds, vmax=vmax)
