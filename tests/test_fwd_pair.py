"""The forward on CTA pairs (fa_fwd_ex with FA_FLAG_CTA_PAIR, head dim 64): two CTAs of a
cluster share every tensor-core product (256 rows; each CTA holds its own 128 rows and half of
every K and V tile). Parity with the fp64 oracle under the forward's tolerances (O max-abs
2e-2, mean-abs 1e-3, LSE 1e-3), on the shapes that exercise its unit of four Q tiles: groups
with fewer than four live tiles (odd and ragged tile counts), tiles past the end of the
sequence, grids smaller than the SM count, and the scale's special values."""

import math

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _pair_fwd(q, k, v, causal, scale=None):
    import torch
    import exact_attention_23_gb300 as fa
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale, flags=fa.FA_FLAG_CTA_PAIR)
    torch.cuda.synchronize()
    return o, lse


def _check(o, lse, o_ref, lse_ref, what, allowance=0.0):
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN + allowance * float(np.abs(o_ref).mean()), f"{what}: O mean-abs {err.mean():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_MAX, f"{what}: LSE max-abs"


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,T", [(1, 3, 777), (1, 2, 128), (2, 12, 1000), (4, 12, 1100), (4, 12, 1153)])
@pytest.mark.parametrize("causal", [True, False])
def test_pair_parity(B, H, T, causal):
    q, k, v = inputs.make_qkv(B, H, T, 64, seed=4000 + T + B)
    o, lse = _pair_fwd(q, k, v, causal)
    o_ref, lse_ref = oracle.attention(inputs.to_f64_numpy(q), inputs.to_f64_numpy(k),
                                      inputs.to_f64_numpy(v), causal, 0.125)
    # shapes outside the named workloads with few keys per row: allow the mean error that
    # rounding O_ref to bf16 alone makes (2^-9 of |O|)
    _check(o, lse, o_ref, lse_ref, f"pair B{B} H{H} T{T} causal={causal}", 2.0 ** -9)


@pytest.mark.gpu
@pytest.mark.parametrize("scale", [-0.125, 0.0])
def test_pair_special_scales(scale):
    q, k, v = inputs.make_qkv(2, 4, 700, 64, seed=4100)
    for causal in (True, False):
        o, lse = _pair_fwd(q, k, v, causal, scale=scale)
        o_ref, lse_ref = oracle.attention(inputs.to_f64_numpy(q), inputs.to_f64_numpy(k),
                                          inputs.to_f64_numpy(v), causal, scale)
        _check(o, lse, o_ref, lse_ref, f"pair scale {scale} causal={causal}", 2.0 ** -9)


@pytest.mark.gpu
@pytest.mark.parametrize("T", [4096, 16384])
def test_pair_sweep_sampled(T):
    """The sweep's workload (B4 H12, seeded as the bench's) on sampled rows of a few heads,
    causal row 0 bit for bit."""
    import torch
    w = inputs.WORKLOADS[f"sweep_t{T}"]
    q, k, v = inputs.workload_qkv(w)
    o, lse = _pair_fwd(q, k, v, True)
    rng = np.random.default_rng(T)
    for bh in (0, 23, 47):
        b, h = divmod(bh, w.H)
        rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, T // 2, T - 1],
                                         rng.integers(0, T, 40)]))
        o_ref, lse_ref = oracle.attention_rows(inputs.to_f64_numpy(q[b, h]), inputs.to_f64_numpy(k[b, h]),
                                               inputs.to_f64_numpy(v[b, h]), True, w.scale, rows)
        idx = torch.from_numpy(rows).cuda()
        _check(o[b, h][idx], lse[b, h][idx], o_ref, lse_ref, f"pair T{T} bh={bh}")
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0]), "causal row 0 must equal v0 bit for bit"
