"""CPU tests of the C ABI's host side: the library loads, exports every symbol the header
declares, and rejects bad arguments before launching anything. No GPU compute here."""

import ctypes
import math
import os
import re

import pytest

import exact_attention_23_gb300 as fa
from exact_attention_23_gb300 import _binding
from tests import oracle_pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    with open(os.path.join(ROOT, "include", "fa.h"), encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_binding.LIB_PATH):
        from exact_attention_23_gb300 import build
        build.build()
    return fa.lib()


def test_header_declares_expected_api():
    assert _header_functions() == sorted(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(lib):
    assert "sm_103a" in fa.version()
    for code in range(6):
        assert fa.strerror(code)
    assert fa.strerror(99) == "unknown status"


def test_status_codes_match_header():
    with open(os.path.join(ROOT, "include", "fa.h"), encoding="utf-8") as f:
        text = f.read()
    for name in ("FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_MISALIGNED", "FA_ERR_UNSUPPORTED_DEVICE",
                 "FA_ERR_LAUNCH", "FA_ERR_TIMEOUT"):
        m = re.search(rf"\b{name}\s*=\s*(\d+)", text)
        assert m and int(m.group(1)) == getattr(fa, name), name
    m = re.search(r"#define\s+FA_FLAG_TEST_STARVE_Q\s+(\d+)u", text)
    assert m and int(m.group(1)) == fa.FA_FLAG_TEST_STARVE_Q
    m = re.search(r"#define\s+FA_FLAG_TEST_STARVE_LATER_Q\s+(\d+)u", text)
    assert m and int(m.group(1)) == fa.FA_FLAG_TEST_STARVE_LATER_Q


# Fake, never-dereferenced device addresses: validation fails before any CUDA call.
A = 0x7F0000000000
SZ = 1 << 30


def _call(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=A + 4 * SZ, B=1, H=1, T=128, d=64,
          causal=1, scale=0.125, flags=0):
    return fa.fa_fwd_ex(q, k, v, o, lse, B, H, T, d, causal, scale, None, 0, flags, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(k=0), fa.FA_ERR_INVALID_ARG),
    (dict(v=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=-1), fa.FA_ERR_INVALID_ARG),
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=3.0e38), fa.FA_ERR_INVALID_ARG),        # scale·log2(e) overflows fp32
    # every finite scale passes validation (0: uniform weights; < 0: reversed preference):
    # these fail only at the misaligned pointer, checked later, before any device call
    (dict(scale=0.0, q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(scale=-0.125, q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(scale=-1.0e30, q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(flags=8), fa.FA_ERR_INVALID_ARG),
    (dict(flags=fa.FA_FLAG_CTA_PAIR, d=128), fa.FA_ERR_INVALID_ARG),   # pairs: head dim 64 only
    (dict(flags=fa.FA_FLAG_CTA_PAIR | fa.FA_FLAG_TEST_STARVE_Q), fa.FA_ERR_INVALID_ARG),
    (dict(flags=fa.FA_FLAG_CTA_PAIR, q=A + 8), fa.FA_ERR_MISALIGNED),  # accepted, then misaligned
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 3 * SZ + 2), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 4 * SZ + 4), fa.FA_ERR_MISALIGNED),
    (dict(o=A), fa.FA_ERR_INVALID_ARG),                 # o aliases q
    (dict(o=A + SZ + 4096), fa.FA_ERR_INVALID_ARG),     # o overlaps k
    (dict(lse=A + 2 * SZ + 16), fa.FA_ERR_INVALID_ARG),  # lse overlaps v
    (dict(B=1 << 16, H=1 << 15, T=1 << 16), fa.FA_ERR_INVALID_ARG),  # grid / size overflow
])
def test_host_validation_rejects_before_launch(lib, kw, want):
    assert _call(**kw) == want


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a machine without a CUDA device")
def test_valid_call_without_device_reports_unsupported(lib):
    assert _call() == fa.FA_ERR_UNSUPPORTED_DEVICE
    assert fa.fa_fwd(A, A + SZ, A + 2 * SZ, A + 3 * SZ, A + 4 * SZ, 1, 1, 128, 64, 1, 0.125,
                     None) == fa.FA_ERR_UNSUPPORTED_DEVICE


def test_python_wrapper_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd(x, x, x)


def test_flop_and_byte_counts():
    # causal FLOPs are half of 4·B·H·T²·d; bytes read q,k,v and write o (bf16) + lse (fp32)
    assert fa.flops(4, 12, 4096, 64, True) == 0.5 * 4 * 4 * 12 * 4096 ** 2 * 64
    assert fa.flops(2, 16, 16384, 128, False) == 4 * 2 * 16 * 16384 ** 2 * 128
    assert fa.hbm_bytes(4, 12, 512, 64) == 24768 * 512


def test_tiling_arithmetic_matches_the_page():
    """The page's grid of (Q blocks, batch·heads) with 64-row blocks gives 3072 programs
    at B4 H12 T4096; the same helper sizes this library's 128-row tiles."""
    facts = oracle_pins.load_page_facts()
    assert fa.q_tiles(4096, 64) * 4 * 12 == facts["programs_b4_h12_t4096_block64"]
    assert fa.q_tiles(1000) == 8 and fa.q_tiles(128) == 1 and fa.q_tiles(129) == 2
    assert math.ceil(fa.q_tiles(4096) / 2) * 48 == 768


# ------------------------------------------------------------------------------ backward

def test_bwd_workspace_size(lib):
    # [BH][T_pad] lse2 and D (fp32) plus a [BH][T_pad][d] fp32 dQ accumulator, 256-aligned
    assert fa.fa_bwd_workspace_size(1, 1, 128, 64) == 2 * 512 + 128 * 64 * 4
    assert fa.fa_bwd_workspace_size(2, 3, 129, 64) == 2 * 6 * 256 * 4 + 6 * 256 * 64 * 4
    assert fa.fa_bwd_workspace_size(4, 12, 16384, 64) == 48 * 16384 * (2 + 64) * 4
    assert fa.fa_bwd_workspace_size(1, 1, 1, 64) == 2 * 512 + 128 * 64 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 128, 128) == 2 * 512 + 128 * 128 * 4
    for bad in ((0, 1, 128, 64), (1, 0, 128, 64), (1, 1, 0, 64), (1, 1, 128, 96),
                (1, 1, 128, 32), (1 << 16, 1 << 15, 1 << 16, 64)):
        assert fa.fa_bwd_workspace_size(*bad) == 0, bad


def _bwd_call(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, do=A + 4 * SZ, lse=A + 5 * SZ,
              dq=A + 6 * SZ, dk=A + 7 * SZ, dv=A + 8 * SZ, ws=A + 9 * SZ, ws_bytes=None, B=1, H=1,
              T=128, d=64, causal=1, scale=0.125, flags=0):
    if ws_bytes is None:
        ws_bytes = max(fa.fa_bwd_workspace_size(B, H, T, 64), 1 << 20)
    return fa.fa_bwd_ex(q, k, v, o, do, lse, dq, dk, dv, ws, ws_bytes, B, H, T, d, causal, scale,
                        None, 0, flags, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(do=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(flags=4), fa.FA_ERR_INVALID_ARG),
    (dict(ws_bytes=1024), fa.FA_ERR_INVALID_ARG),                   # workspace too small
    (dict(ws=A + 9 * SZ + 16), fa.FA_ERR_MISALIGNED),               # workspace not 256-aligned
    (dict(dk=A + 7 * SZ + 8), fa.FA_ERR_MISALIGNED),
    (dict(dq=A), fa.FA_ERR_INVALID_ARG),                            # dq aliases q
    (dict(dv=A + 6 * SZ + 4096), fa.FA_ERR_INVALID_ARG),            # dv overlaps dq
    (dict(ws=A + 5 * SZ), fa.FA_ERR_INVALID_ARG),                   # workspace overlaps lse
])
def test_bwd_host_validation_rejects_before_launch(lib, kw, want):
    assert _bwd_call(**kw) == want


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a machine without a CUDA device")
def test_bwd_valid_call_without_device_reports_unsupported(lib):
    assert _bwd_call() == fa.FA_ERR_UNSUPPORTED_DEVICE


def test_bwd_flop_count():
    assert fa.bwd_flops(4, 12, 4096, 64, True) == 2.5 * fa.flops(4, 12, 4096, 64, True)



def test_library_exports_only_the_c_abi(lib):
    """libfa.so exports exactly the functions include/fa.h declares (a linker version
    script hides everything else)."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", _binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    funcs = sorted(line.split()[-1] for line in out.splitlines()
                   if len(line.split()) == 3 and line.split()[1] == "T")
    assert funcs == _header_functions()


# ---------------------------------------------------------------- general forward forms

def _kv_call(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=A + 4 * SZ, B=1, H=2, Tq=1, Tk=1000,
             d=64, causal=1, scale=0.125, n_splits=1, ws=None, ws_bytes=0):
    return fa.fa_fwd_kv(q, k, v, o, lse, B, H, Tq, Tk, d, causal, scale, n_splits, ws, ws_bytes,
                        None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(Tq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Tk=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_INVALID_ARG),
    (dict(Tq=2000, Tk=1000), fa.FA_ERR_INVALID_ARG),      # causal needs Tq <= Tk
    (dict(n_splits=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(o=A + 3 * SZ + 2), fa.FA_ERR_MISALIGNED),
    (dict(o=A + SZ), fa.FA_ERR_INVALID_ARG),              # o aliases k
])
def test_fwd_kv_host_validation(lib, kw, want):
    assert _kv_call(**kw) == want


def test_fwd_kv_workspace_size(lib):
    # explicit splits: S·B·H·Tq·d·4 bytes of partial O plus S·B·H·Tq·4 of LSE, 256-aligned
    assert fa.fa_fwd_kv_workspace_size(2, 12, 1, 4096, 64, 4) == (
        -(-4 * 24 * 64 * 4 // 256) * 256 + -(-4 * 24 * 4 // 256) * 256)
    assert fa.fa_fwd_kv_workspace_size(2, 12, 1, 4096, 64, 1) == 1   # no workspace needed
    assert fa.fa_fwd_kv_workspace_size(1, 1, 3, 100, 64, 8) == 1     # one K tile: one range
    # two query rows run on the CUDA cores, whose key ranges count keys, not K tiles:
    # 8 ranges of 13 keys, S·B·H·Tq·d·4 + S·B·H·Tq·4 bytes, 256-aligned
    assert fa.fa_fwd_kv_workspace_size(1, 1, 2, 100, 64, 8) == 8 * 2 * 64 * 4 + 256
    # one query row (decode): ranges are counted in keys; 100 keys in 8 ranges of 13
    assert fa.fa_fwd_kv_workspace_size(1, 1, 1, 100, 64, 8) == 8 * 64 * 4 // 256 * 256 + 256
    assert fa.fa_fwd_kv_workspace_size(1, 1, 1, 3, 64, 8) == 3 * 64 * 4 + 256  # at most Tk ranges
    assert fa.fa_fwd_kv_workspace_size(1, 1, 0, 100, 64, 2) == 0
    assert fa.fa_fwd_kv_workspace_size(1, 1, 1, 100, 32, 2) == 0


def _bs_call(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=A + 4 * SZ, mask=A + 5 * SZ,
             mask_heads=1, B=1, H=2, T=1000, d=64, causal=0, scale=0.125):
    return fa.fa_fwd_block_sparse(q, k, v, o, lse, mask, mask_heads, B, H, T, d, causal, scale,
                                  None)


@pytest.mark.parametrize("kw,want", [
    (dict(mask=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask_heads=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask_heads=3), fa.FA_ERR_INVALID_ARG),           # neither 1 nor B·H
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=256), fa.FA_ERR_INVALID_ARG),
    (dict(lse=A + 4 * SZ + 4), fa.FA_ERR_MISALIGNED),
])
def test_fwd_block_sparse_host_validation(lib, kw, want):
    assert _bs_call(**kw) == want


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a machine without a CUDA device")
def test_general_forms_without_device_report_unsupported(lib):
    assert _kv_call() == fa.FA_ERR_UNSUPPORTED_DEVICE
    assert _bs_call() == fa.FA_ERR_UNSUPPORTED_DEVICE
    assert _bs_call(mask_heads=2) == fa.FA_ERR_UNSUPPORTED_DEVICE
    assert fa.fa_fwd_kv_workspace_size(1, 1, 1, 1000, 64, 0) == 0   # automatic choice needs a device


# ---------------------------------------------------------------- FP8 (e4m3) query/key forward

def _fp8_call(q8=A, k8=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=A + 4 * SZ, q_scale=0.01,
              k_scale=0.02, B=1, H=2, T=1000, d=64, causal=1, scale=0.125):
    return fa.fa_fwd_fp8(q8, k8, v, o, lse, q_scale, k_scale, B, H, T, d, causal, scale, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q8=0), fa.FA_ERR_INVALID_ARG),
    (dict(k8=0), fa.FA_ERR_INVALID_ARG),
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_INVALID_ARG),
    (dict(q_scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(k_scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(q_scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q8=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=A + SZ + 4096), fa.FA_ERR_INVALID_ARG),     # o overlaps the codes of k
])
def test_fwd_fp8_host_validation(lib, kw, want):
    assert _fp8_call(**kw) == want


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a machine without a CUDA device")
def test_fwd_fp8_without_device_reports_unsupported(lib):
    assert _fp8_call() == fa.FA_ERR_UNSUPPORTED_DEVICE
    # o directly after q's one-byte codes does not overlap them
    assert _fp8_call(o=A + 2 * 1000 * 64) == fa.FA_ERR_UNSUPPORTED_DEVICE


def test_fwd_fp8_wrapper_rejects_bf16_codes():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fwd_fp8(x, 1.0, x, 1.0, x)


# ---------------------------------------------------------------- host-memory forward

def _host_call(q=A, k=A + SZ, v=A + 2 * SZ, o=A + 3 * SZ, lse=A + 4 * SZ, B=1, H=4, T=1000,
               d=64, causal=1, scale=0.125, hpc=2, ws=A + 5 * SZ, ws_bytes=1 << 30):
    return fa.fa_fwd_host(q, k, v, o, lse, B, H, T, d, causal, scale, hpc, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(ws=0), fa.FA_ERR_INVALID_ARG),
    (dict(T=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_INVALID_ARG),
    (dict(hpc=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(ws=A + 5 * SZ + 128), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 4096), fa.FA_ERR_INVALID_ARG),            # o overlaps q
    (dict(ws_bytes=1024), fa.FA_ERR_INVALID_ARG),          # workspace too small
])
def test_fwd_host_validation(lib, kw, want):
    assert _host_call(**kw) == want


def test_fwd_host_workspace_size(lib):
    # three staging buffers of c heads: q, k, v, o (bf16) and lse (fp32), each 256-aligned
    def chunk(c, T, d):
        r = lambda x: -(-x // 256) * 256
        return 4 * r(c * T * d * 2) + r(c * T * 4)
    assert fa.fa_fwd_host_workspace_size(2, 6, 1000, 64, 4) == 3 * chunk(4, 1000, 64)
    assert fa.fa_fwd_host_workspace_size(2, 6, 1000, 128, 100) == 3 * chunk(12, 1000, 128)
    assert fa.fa_fwd_host_workspace_size(2, 6, 1000, 96, 4) == 0
    assert fa.fa_fwd_host_workspace_size(2, 6, 1000, 64, -1) == 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="only meaningful on a machine without a CUDA device")
def test_fwd_host_without_device_reports_unsupported(lib):
    assert _host_call() == fa.FA_ERR_UNSUPPORTED_DEVICE
    assert _host_call(hpc=0) == fa.FA_ERR_UNSUPPORTED_DEVICE    # automatic chunking
    assert fa.fa_fwd_host_workspace_size(1, 4, 1000, 64, 0) == 0


def test_fwd_host_wrapper_rejects_device_or_wrong_dtype():
    import torch
    x = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(ValueError):
        fa.fwd_host(x, x, x)
