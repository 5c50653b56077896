"""GPU parity at the sizes, seeds and launch configuration of bench.py's secondary objects
(decode, a few new queries, block-sparse, FP8), against the fp64 oracle: every head where the
oracle is cheap (decode and a few queries: one to 128 query rows per head), otherwise whole
heads picked from the batch (block-sparse) or sampled rows (FP8). Tolerances as for the forward: O max-abs ≤ 2e-2, mean-abs ≤ 1e-3,
LSE ≤ 1e-3."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _check(o, lse, o_ref, lse_ref, what, mean_allow=0.0):
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), what
    assert err.max() <= O_MAX, f"{what}: O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN + mean_allow, f"{what}: O mean-abs {err.mean():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_MAX, f"{what}: LSE"


def test_decode_bench_size_every_head():
    """B4 H12 d64: the query is the last of a T = 16384 draw (seed 20) against all 16384
    keys, causal, automatic key ranges (as the bench times it)."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, Tk, d = 4, 12, 16384, 64
    q, k, v = inputs.make_qkv(B, H, Tk, d, seed=20)
    q1 = q[:, :, -1:].contiguous()
    o, lse = fa.fwd_kv(q1.cuda(), k.cuda(), v.cuda(), causal=True, n_splits=0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_general(*(inputs.to_f64_numpy(t) for t in (q1, k, v)),
                                              True, d ** -0.5)
    # one row per head sees 16384 keys: |O| is small; rounding allowance as for short rows
    _check(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
           "decode B4 H12 Tk16384", 2.0 ** -9 * float(np.abs(o_ref).mean()))


@pytest.mark.parametrize("tq", [2, 8, 128])
def test_few_queries_bench_size_every_head(tq):
    """B4 H12 d64: the last tq queries of the decode object's T = 16384 draw (seed 20) against
    all 16384 keys, bottom-right causal, automatic key ranges (bench.py's
    fwd_kv_few_queries): Tq = 2 on the CUDA-core multi-query kernel, 8 and 128 on the
    one-tile general form with split ranges."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, Tk, d = 4, 12, 16384, 64
    q, k, v = inputs.make_qkv(B, H, Tk, d, seed=20)
    qm = q[:, :, -tq:].contiguous()
    o, lse = fa.fwd_kv(qm.cuda(), k.cuda(), v.cuda(), causal=True, n_splits=0)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention_general(*(inputs.to_f64_numpy(t) for t in (qm, k, v)),
                                              True, d ** -0.5)
    _check(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
           f"few queries Tq{tq} B4 H12 Tk16384", 2.0 ** -9 * float(np.abs(o_ref).mean()))


def test_block_sparse_bench_size_two_heads():
    """B4 H12 T8192 d64, non-causal, the bench's seeded mask (generator seed 22, half the
    128×128 blocks kept); heads (0, 0) and (3, 11) checked in full against the oracle."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 4, 12, 8192, 64
    q, k, v = inputs.make_qkv(B, H, T, d, seed=21)
    nb = fa.q_tiles(T)
    g = torch.Generator(device="cpu")
    g.manual_seed(22)
    mask = (torch.rand((nb, nb), generator=g) < 0.5).to(torch.uint8)
    o, lse = fa.fwd_block_sparse(q.cuda(), k.cuda(), v.cuda(), mask.cuda().contiguous(),
                                 causal=False)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    for b, h in ((0, 0), (3, 11)):
        o_ref, lse_ref = oracle.attention_general_head(
            *(inputs.to_f64_numpy(t[b, h]) for t in (q, k, v)), False, d ** -0.5,
            mask.numpy())
        _check(o[b, h], lse[b, h], o_ref, lse_ref, f"block-sparse head ({b},{h})")


def test_fp8_bench_size_sampled_rows():
    """B2 H16 T16384 d128 causal, e4m3 q/k of the seed-30 draw, bf16 v; rows sampled in
    two heads."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 2, 16, 16384, 128
    q8, sq, k8, sk, v = inputs.make_qk_fp8(B, H, T, d, seed=30)
    o, lse = fa.fwd_fp8(q8.cuda(), sq, k8.cuda(), sk, v.cuda(), causal=True)
    torch.cuda.synchronize()
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    qd, kd = inputs.dequantize_e4m3(q8, sq), inputs.dequantize_e4m3(k8, sk)
    vd = inputs.to_f64_numpy(v)
    rows = np.array(sorted({0, 127, 128, 8191, 8192, T - 1} |
                           set(np.random.default_rng(6).integers(0, T, 16).tolist())))
    for b, h in ((0, 0), (1, 15)):
        o_ref, lse_ref = oracle.attention_rows(qd[b, h], kd[b, h], vd[b, h], True, d ** -0.5,
                                               rows)
        _check(o[b, h, rows], lse[b, h, rows], o_ref, lse_ref, f"fp8 head ({b},{h})")
