"""GPU parity of the FP8 query/key forward (fa_fwd_fp8) against the fp64 oracle.

Q and K are e4m3 codes with per-tensor scales (inputs.make_qk_fp8: the bf16 workload draw,
quantised); the oracle runs plain attention on the exact values those codes stand for
(dequantize_e4m3), with the bf16 V. The kernel's scores are exact products of the codes
summed in fp32, so the comparison carries the same error sources as the bf16 forward (fp32
sums, P rounded to bf16 for P·V, bf16 output) and takes the forward's tolerances: O max-abs
≤ 2e-2, mean-abs ≤ 1e-3, LSE max-abs ≤ 1e-3."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _run(B, H, T, d, causal, seed):
    import torch
    import exact_attention_23_gb300 as fa
    q8, sq, k8, sk, v = inputs.make_qk_fp8(B, H, T, d, seed)
    o, lse = fa.fwd_fp8(q8.cuda(), sq, k8.cuda(), sk, v.cuda(), causal=causal)
    torch.cuda.synchronize()
    return (q8, sq, k8, sk, v), o.float().cpu().double().numpy(), lse.cpu().double().numpy()


@pytest.mark.parametrize("B,H,T,d,causal", [
    (1, 2, 128, 64, True),      # one tile
    (2, 3, 1000, 64, True),     # several tiles, ragged tail
    (2, 3, 1000, 64, False),
    (1, 4, 777, 128, True),
    (2, 2, 1024, 128, False),
    (1, 1, 1, 64, True),        # a single row
    (1, 2, 129, 128, True),     # one row past a tile
])
def test_fwd_fp8_parity(B, H, T, d, causal):
    (q8, sq, k8, sk, v), o, lse = _run(B, H, T, d, causal, 900 + T + d)
    qd, kd = inputs.dequantize_e4m3(q8, sq), inputs.dequantize_e4m3(k8, sk)
    o_ref, lse_ref = oracle.attention(qd, kd, inputs.to_f64_numpy(v), causal, d ** -0.5)
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"O mean-abs {err.mean():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_MAX


def test_fwd_fp8_sampled_rows_at_length_16384():
    """T = 16384, d = 64, causal: rows sampled across the sequence (first, last, tile edges
    and random) against the oracle's row-by-row form."""
    B, H, T, d = 1, 2, 16384, 64
    (q8, sq, k8, sk, v), o, lse = _run(B, H, T, d, True, 77)
    qd, kd = inputs.dequantize_e4m3(q8, sq), inputs.dequantize_e4m3(k8, sk)
    vd = inputs.to_f64_numpy(v)
    rows = sorted({0, 1, 127, 128, 8191, 8192, T - 1} |
                  set(np.random.default_rng(5).integers(0, T, 24).tolist()))
    for b in range(B):
        for h in range(H):
            o_ref, lse_ref = oracle.attention_rows(qd[b, h], kd[b, h], vd[b, h], True, d ** -0.5,
                                                   np.array(rows))
            err = np.abs(o[b, h, rows] - o_ref)
            assert err.max() <= O_MAX, f"(b{b} h{h}) O max-abs {err.max():.3e}"
            assert np.abs(lse[b, h, rows] - lse_ref).max() <= LSE_MAX


def test_fwd_fp8_matches_bf16_forward_on_the_same_values():
    """The e4m3 values are exact in bf16, so the bf16 forward on the dequantised, rescaled
    inputs computes the same attention: outputs agree to the forward's tolerance."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 2, 4, 2048, 128
    q8, sq, k8, sk, v = inputs.make_qk_fp8(B, H, T, d, 31)
    qb = q8.view(torch.float8_e4m3fn).to(torch.bfloat16).cuda()
    kb = k8.view(torch.float8_e4m3fn).to(torch.bfloat16).cuda()
    o8, l8 = fa.fwd_fp8(q8.cuda(), sq, k8.cuda(), sk, v.cuda(), causal=True)
    ob, lb = fa.fwd(qb, kb, v.cuda(), causal=True, scale=d ** -0.5 * sq * sk)
    torch.cuda.synchronize()
    assert (o8.float() - ob.float()).abs().max().item() <= O_MAX
    assert (l8 - lb).abs().max().item() <= LSE_MAX
