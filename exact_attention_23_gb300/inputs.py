"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle checks.

This module holds no attention arithmetic: it only draws q, k, v. Both sides of every
parity test consume the same bf16 buffers made here.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws q, then k, then
v with ``randn`` in fp32 (shape [B, H, T, d]); each is multiplied by ``std`` and cast to
bf16 with round-to-nearest-even. For the "spiky" workload one key row per (b, h),
at an index drawn afterwards from the same generator uniformly in [128, T), is
multiplied by 8 in fp32 before the cast, so that every query that sees that key meets
a large jump of the running row max in the middle of its scan. The upstream gradient dO
of a backward test comes from a second generator seeded with seed + 1_000_003, drawn
with ``randn`` in fp32 and cast to bf16 the same way. The pages' workloads
use random bf16 q/k/v at GPT-2 124M head shapes (12 heads of width 64) and a length
sweep up to 16k ("Hand-written FlashAttention", steps ④ and ⑤).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    causal: bool
    seed: int
    std: float = 1.0
    spike: str | None = None   # None, "k" or "q": which tensor gets one ×8 row per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_causal(self, causal: bool) -> "Workload":
        return Workload(self.name, self.B, self.H, self.T, self.d, causal, self.seed,
                        self.std, self.spike)


SWEEP_T = (512, 1024, 2048, 4096, 8192, 16384)

WORKLOADS = {
    "tiny_causal": Workload("tiny_causal", 1, 2, 256, 64, True, 0),
    "ragged_t1000": Workload("ragged_t1000", 2, 12, 1000, 64, True, 1),
    "gpt2_layer_spiky": Workload("gpt2_layer_spiky", 4, 12, 1024, 64, True, 2, 0.5, "k"),
    "gpt2_layer_spiky_q": Workload("gpt2_layer_spiky_q", 4, 12, 1024, 64, True, 2, 0.5, "q"),
    "wide_head_t16k": Workload("wide_head_t16k", 2, 16, 16384, 128, True, 10),
}
for _i, _t in enumerate(SWEEP_T):
    WORKLOADS[f"sweep_t{_t}"] = Workload(f"sweep_t{_t}", 4, 12, _t, 64, True, 3 + _i)


def make_qkv(B: int, H: int, T: int, d: int, seed: int, std: float = 1.0,
             spike: str | None = None):
    """Draw (q, k, v) as contiguous bf16 CPU tensors of shape [B, H, T, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (B, H, T, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        q.mul_(std)
        k.mul_(std)
        v.mul_(std)
    if spike is not None:
        if T <= 128:
            raise ValueError("a spiky workload needs T > 128")
        rows = torch.randint(128, T, (B, H), generator=g)
        target = {"k": k, "q": q}[spike]
        for b in range(B):
            for h in range(H):
                target[b, h, int(rows[b, h])] *= 8.0
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def workload_qkv(w: Workload):
    return make_qkv(w.B, w.H, w.T, w.d, w.seed, w.std, w.spike)


def to_f64_numpy(t: torch.Tensor):
    """Exact bf16 → fp64 numpy view for the oracle (bf16 values are exact in fp64)."""
    return t.detach().to("cpu", torch.float64).numpy()


def make_do(B: int, H: int, T: int, d: int, seed: int):
    """Draw the upstream gradient dO ([B, H, T, d] bf16, standard normal) for a backward
    test of the workload with this seed."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1_000_003)
    return torch.randn((B, H, T, d), generator=g, dtype=torch.float32).to(torch.bfloat16).contiguous()


def workload_do(w: Workload):
    return make_do(w.B, w.H, w.T, w.d, w.seed)


E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor FP8 (e4m3) quantisation of an input: scale = max|x| / 448, codes =
    round-to-nearest-even of x / scale. Returns (codes as a uint8 tensor of x's shape,
    scale as a Python float); the value a code stands for is e4m3(code) · scale."""
    x = x.float()
    amax = float(x.abs().max())
    # a float32 value, so the scale handed to the C ABI is exactly the one the codes use
    scale = torch.tensor(amax / E4M3_MAX, dtype=torch.float32).item() if amax > 0 else 1.0
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, scale


def dequantize_e4m3(codes: torch.Tensor, scale: float):
    """The exact values of e4m3 codes times the scale, as fp64 numpy (every e4m3 value and
    its product with a float scale is exact in fp64)."""
    return codes.view(torch.float8_e4m3fn).double().numpy() * scale


def make_qk_fp8(B: int, H: int, T: int, d: int, seed: int):
    """The workload's q and k (make_qkv with this seed) quantised to e4m3 per tensor, and its
    v in bf16: (q8, q_scale, k8, k_scale, v)."""
    q, k, v = make_qkv(B, H, T, d, seed)
    q8, sq = quantize_e4m3(q)
    k8, sk = quantize_e4m3(k)
    return q8, sq, k8, sk, v
