"""Seeded randomised parity of the forward entry points against plain PyTorch fp32 math on
the GPU (softmax(scale·QKᵀ + mask)·V and its logsumexp), over shapes the named workloads do
not reach: random batch and head counts, ragged lengths on both sides of the short-grid
switch, both head dims, causal or not, scales of either sign, and for the general forms
random query/key lengths, key-range counts and block masks; the FP8 forward against the
values its e4m3 codes stand for, and the forward on CTA pairs. Tolerances: O mean-abs ≤ 1e-3 +
2⁻⁹·mean|O_ref| and LSE ≤ 1e-3 on rows that see a key, as for the oracle tests; O max-abs ≤
max(2e-2, 2⁻⁸·max|V| + 2⁻⁹·max|O_ref| + 1e-3). The kernels round each probability to bf16
(relative error ≤ 2⁻⁸) before P·V, which moves O_i by at most 2⁻⁸·Σ_j p_ij·|v_j| / l_i ≤
2⁻⁸·max|V|, and round O to bf16 (≤ 2⁻⁹·|O|); a large |scale| (a peaked softmax over
few keys) brings the first term close to its bound. Rows that see no key must be O = 0,
LSE = −∞."""

import numpy as np
import pytest

from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 1e-3, 1e-3


def _ref(q, k, v, scale, mask):
    """fp32 reference on the GPU: mask is a boolean [Tq, Tk] (True = visible) or None."""
    import torch
    s = torch.matmul(q.float(), k.float().transpose(-1, -2)) * scale
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.softmax(s, dim=-1)
    p = torch.nan_to_num(p, nan=0.0)  # rows that see no key
    return torch.matmul(p, v.float()), lse


def _check(o, lse, o_ref, lse_ref, what, v):
    import torch
    o, o_ref = o.float(), o_ref.float()
    o_max = max(O_MAX, 2.0 ** -8 * v.float().abs().max().item()
                + 2.0 ** -9 * o_ref.abs().max().item() + 1e-3)
    live = torch.isfinite(lse_ref)
    assert bool(torch.isfinite(o).all()), f"{what}: non-finite O"
    assert bool(torch.equal(torch.isneginf(lse), ~live)), f"{what}: empty rows differ"
    assert bool((o[~live] == 0).all()), f"{what}: empty rows must be 0"
    err = (o - o_ref).abs()
    assert err.max().item() <= o_max, f"{what}: O max-abs {err.max().item():.3e} > {o_max:.3e}"
    bound = O_MEAN + 2.0 ** -9 * o_ref.abs().mean().item()
    assert err.mean().item() <= bound, f"{what}: O mean-abs {err.mean().item():.3e}"
    if bool(live.any()):
        lerr = (lse[live] - lse_ref[live]).abs().max().item()
        assert lerr <= LSE_MAX, f"{what}: LSE max-abs {lerr:.3e}"


@pytest.mark.parametrize("case", range(40))
def test_fuzz_dense_forward(case):
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(9000 + case)
    B, H = int(rng.integers(1, 5)), int(rng.integers(1, 17))
    T = int(rng.choice([int(rng.integers(1, 400)), int(rng.integers(400, 3000))]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.choice([d ** -0.5, -0.1, 0.3, 0.0]))
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, T, d, 9100 + case))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    mask = torch.ones(T, T, dtype=torch.bool, device="cuda").tril() if causal else None
    o_ref, lse_ref = _ref(q, k, v, scale, mask)
    _check(o, lse, o_ref, lse_ref, f"fwd B{B} H{H} T{T} d{d} causal={causal} scale={scale}", v)


@pytest.mark.parametrize("case", range(40))
def test_fuzz_fwd_kv(case):
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(9200 + case)
    B, H = int(rng.integers(1, 5)), int(rng.integers(1, 13))
    Tk = int(rng.integers(1, 6000))
    Tq = int(rng.choice([1, 2, int(rng.integers(3, 129)), int(rng.integers(1, Tk + 1))]))
    Tq = min(Tq, Tk)
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    n_splits = int(rng.choice([0, 0, 1, int(rng.integers(2, 9))]))
    scale = float(rng.choice([d ** -0.5, -0.2]))
    q, k, v = inputs.make_qkv(B, H, Tk, d, 9300 + case)
    q = q[:, :, Tk - Tq:].contiguous()
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.fwd_kv(q, k, v, causal=causal, scale=scale, n_splits=n_splits)
    mask = None
    if causal:  # bottom-right: query i sees keys j ≤ i + Tk − Tq
        i = torch.arange(Tq, device="cuda")[:, None]
        j = torch.arange(Tk, device="cuda")[None, :]
        mask = j <= i + (Tk - Tq)
    o_ref, lse_ref = _ref(q, k, v, scale, mask)
    _check(o, lse, o_ref, lse_ref,
           f"fwd_kv B{B} H{H} Tq{Tq} Tk{Tk} d{d} causal={causal} splits={n_splits} scale={scale}", v)


@pytest.mark.parametrize("case", range(24))
def test_fuzz_block_sparse(case):
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(9400 + case)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 9))
    T = int(rng.integers(1, 3000))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    per_head = bool(rng.integers(0, 2))
    density = float(rng.choice([0.1, 0.5, 0.9]))
    nb = -(-T // 128)
    heads = B * H if per_head else 1
    m = (rng.random((heads, nb, nb)) < density).astype(np.uint8)
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, T, d, 9500 + case))
    mt = torch.from_numpy(m if per_head else m[0]).cuda().contiguous()
    o, lse = fa.fwd_block_sparse(q, k, v, mt, causal=causal)
    # element mask: block mask expanded to keys and queries, and causal on top
    bm = torch.from_numpy(m).cuda().bool()
    full = bm.repeat_interleave(128, dim=1).repeat_interleave(128, dim=2)[:, :T, :T]
    if causal:
        full = full & torch.ones(T, T, dtype=torch.bool, device="cuda").tril()
    full = full.reshape(B, H, T, T) if per_head else full[0]
    o_ref, lse_ref = _ref(q, k, v, d ** -0.5, full)
    _check(o, lse, o_ref, lse_ref,
           f"block-sparse B{B} H{H} T{T} d{d} causal={causal} per_head={per_head} density={density}", v)


@pytest.mark.parametrize("case", range(24))
def test_fuzz_backward(case):
    """fa_bwd on random shapes against fp32 PyTorch autograd on the GPU, with the
    scale-relative bounds of the sampled backward checks (max|G − G_ref| ≤ 2e-2·max|G_ref|,
    mean ≤ 5e-3·mean|G_ref|): the kernel rounds P and dS to bf16 before their products."""
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(9600 + case)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 9))
    T = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 2000))]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.choice([d ** -0.5, 0.05, -0.1]))
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, T, d, 9700 + case))
    do = inputs.make_do(B, H, T, d, 9700 + case).cuda()
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    qf, kf, vf = (t.float().requires_grad_(True) for t in (q, k, v))
    s = torch.matmul(qf, kf.transpose(-1, -2)) * scale
    if causal:
        s = s.masked_fill(~torch.ones(T, T, dtype=torch.bool, device="cuda").tril(), float("-inf"))
    torch.matmul(torch.softmax(s, dim=-1), vf).backward(do.float())
    what = f"bwd B{B} H{H} T{T} d{d} causal={causal} scale={scale}"
    for name, g, r in (("dQ", dq, qf.grad), ("dK", dk, kf.grad), ("dV", dv, vf.grad)):
        g, r = g.float(), r.float()
        assert bool(torch.isfinite(g).all()), f"{what}: {name} not finite"
        err = (g - r).abs()
        assert err.max().item() <= 2e-2 * r.abs().max().item() + 1e-6, \
            f"{what}: {name} max-abs {err.max().item():.3e} (max|ref| {r.abs().max().item():.3e})"
        assert err.mean().item() <= 5e-3 * r.abs().mean().item() + 1e-6, \
            f"{what}: {name} mean-abs {err.mean().item():.3e} (mean|ref| {r.abs().mean().item():.3e})"


@pytest.mark.parametrize("case", range(16))
def test_fuzz_fp8(case):
    """fa_fwd_fp8 (e4m3 query/key codes with per-tensor scales, bf16 V) against fp32 math on
    the values the codes stand for."""
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(9800 + case)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 13))
    T = int(rng.choice([int(rng.integers(1, 400)), int(rng.integers(400, 3000))]))
    d = int(rng.choice([64, 128]))
    causal = bool(rng.integers(0, 2))
    q8, sq, k8, sk, v = inputs.make_qk_fp8(B, H, T, d, 9900 + case)
    o, lse = fa.fwd_fp8(q8.cuda(), sq, k8.cuda(), sk, v.cuda(), causal=causal)
    qf = q8.cuda().view(torch.float8_e4m3fn).float() * sq
    kf = k8.cuda().view(torch.float8_e4m3fn).float() * sk
    mask = torch.ones(T, T, dtype=torch.bool, device="cuda").tril() if causal else None
    o_ref, lse_ref = _ref(qf, kf, v.cuda(), d ** -0.5, mask)
    _check(o, lse, o_ref, lse_ref, f"fp8 B{B} H{H} T{T} d{d} causal={causal}", v)


@pytest.mark.parametrize("case", range(16))
def test_fuzz_cta_pair(case):
    """The forward on CTA pairs (FA_FLAG_CTA_PAIR, head dim 64) on random shapes."""
    import torch
    import exact_attention_23_gb300 as fa
    rng = np.random.default_rng(10000 + case)
    B, H = int(rng.integers(1, 5)), int(rng.integers(1, 17))
    T = int(rng.choice([int(rng.integers(1, 600)), int(rng.integers(600, 4000))]))
    causal = bool(rng.integers(0, 2))
    scale = float(rng.choice([0.125, -0.1]))
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, T, 64, 10100 + case))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale, flags=fa.FA_FLAG_CTA_PAIR)
    mask = torch.ones(T, T, dtype=torch.bool, device="cuda").tril() if causal else None
    o_ref, lse_ref = _ref(q, k, v, scale, mask)
    _check(o, lse, o_ref, lse_ref, f"pair B{B} H{H} T{T} causal={causal} scale={scale}", v)
