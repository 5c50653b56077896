"""ctypes binding of libfa.so (include/fa.h), with the same names as the C ABI.

Argument marshalling only: every step of the attention computation runs in the CUDA
kernels of libfa.so. PyTorch is used to own device memory and to name the stream.
There is no fallback: if the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_MISALIGNED = 2
FA_ERR_UNSUPPORTED_DEVICE = 3
FA_ERR_LAUNCH = 4
FA_ERR_TIMEOUT = 5
FA_FLAG_TEST_STARVE_Q = 1
FA_FLAG_TEST_STARVE_LATER_Q = 2
FA_FLAG_CTA_PAIR = 4
FA_BWD_NOALLOC_SCRATCH_BYTES = 33554432

# Every symbol include/fa.h declares.
EXPORTS = ("fa_fwd", "fa_fwd_ex", "fa_fwd_fp8", "fa_fwd_host_workspace_size", "fa_fwd_host", "fa_fwd_kv_workspace_size", "fa_fwd_kv",
           "fa_fwd_block_sparse", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_ex",
           "fa_bwd_noalloc", "fa_strerror", "fa_version")

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({strerror(status)})")


def lib() -> ctypes.CDLL:
    """Load libfa.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with exact_attention_23_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            L.fa_fwd.restype = i
            L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp,
                                    ctypes.c_ulonglong, ctypes.c_uint, vp]
            L.fa_fwd_ex.restype = i
            sz = ctypes.c_size_t
            L.fa_fwd_fp8.argtypes = [vp] * 5 + [f, f, i, i, i, i, i, f, vp]
            L.fa_fwd_host_workspace_size.argtypes = [i, i, i, i, i]
            L.fa_fwd_host_workspace_size.restype = sz
            L.fa_fwd_host.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp, sz, vp]
            L.fa_fwd_host.restype = i
            L.fa_fwd_fp8.restype = i
            L.fa_fwd_kv_workspace_size.argtypes = [i, i, i, i, i, i]
            L.fa_fwd_kv_workspace_size.restype = sz
            L.fa_fwd_kv.argtypes = [vp] * 5 + [i, i, i, i, i, i, f, i, vp, sz, vp]
            L.fa_fwd_kv.restype = i
            L.fa_fwd_block_sparse.argtypes = [vp] * 6 + [i, i, i, i, i, i, f, vp]
            L.fa_fwd_block_sparse.restype = i
            L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
            L.fa_bwd_workspace_size.restype = sz
            L.fa_bwd.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, vp]
            L.fa_bwd.restype = i
            L.fa_bwd_ex.argtypes = [vp] * 10 + [sz, i, i, i, i, i, f, vp, ctypes.c_ulonglong,
                                                ctypes.c_uint, vp]
            L.fa_bwd_ex.restype = i
            L.fa_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, f, vp]
            L.fa_bwd_noalloc.restype = i
            L.fa_strerror.argtypes = [i]
            L.fa_strerror.restype = ctypes.c_char_p
            L.fa_version.argtypes = []
            L.fa_version.restype = ctypes.c_char_p
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def version() -> str:
    return lib().fa_version().decode()


def fa_fwd(q, k, v, o, lse, B, H, T, d, causal, scale, stream) -> int:
    """Raw call: integer addresses in, status out."""
    return lib().fa_fwd(q, k, v, o, lse, B, H, T, d, int(bool(causal)), float(scale), stream)


def fa_fwd_ex(q, k, v, o, lse, B, H, T, d, causal, scale, status, timeout_ns, flags,
              stream) -> int:
    return lib().fa_fwd_ex(q, k, v, o, lse, B, H, T, d, int(bool(causal)), float(scale),
                           status, int(timeout_ns), int(flags), stream)


def fa_bwd_workspace_size(B, H, T, d) -> int:
    return int(lib().fa_bwd_workspace_size(B, H, T, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, T, d, causal,
           scale, stream) -> int:
    return lib().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, int(workspace_bytes), B,
                        H, T, d, int(bool(causal)), float(scale), stream)


def fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, T, d,
              causal, scale, status, timeout_ns, flags, stream) -> int:
    return lib().fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, int(workspace_bytes),
                           B, H, T, d, int(bool(causal)), float(scale), status,
                           int(timeout_ns), int(flags), stream)


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, T, d, causal, scale, stream) -> int:
    return lib().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, T, d,
                                int(bool(causal)), float(scale), stream)


def fa_fwd_kv_workspace_size(B, H, Tq, Tk, d, n_splits) -> int:
    return int(lib().fa_fwd_kv_workspace_size(B, H, Tq, Tk, d, n_splits))


def fa_fwd_kv(q, k, v, o, lse, B, H, Tq, Tk, d, causal, scale, n_splits, workspace,
              workspace_bytes, stream) -> int:
    return lib().fa_fwd_kv(q, k, v, o, lse, B, H, Tq, Tk, d, int(bool(causal)), float(scale),
                           int(n_splits), workspace, int(workspace_bytes), stream)


def fa_fwd_block_sparse(q, k, v, o, lse, block_mask, mask_heads, B, H, T, d, causal, scale,
                        stream) -> int:
    return lib().fa_fwd_block_sparse(q, k, v, o, lse, block_mask, int(mask_heads), B, H, T, d,
                                     int(bool(causal)), float(scale), stream)


def fa_fwd_fp8(q8, k8, v, o, lse, q_scale, k_scale, B, H, T, d, causal, scale, stream) -> int:
    return lib().fa_fwd_fp8(q8, k8, v, o, lse, float(q_scale), float(k_scale), B, H, T, d,
                            int(bool(causal)), float(scale), stream)


def fa_fwd_host_workspace_size(B, H, T, d, heads_per_chunk=0) -> int:
    return int(lib().fa_fwd_host_workspace_size(B, H, T, d, heads_per_chunk))


def fa_fwd_host(q, k, v, o, lse, B, H, T, d, causal, scale, heads_per_chunk, ws, ws_bytes,
                stream) -> int:
    return lib().fa_fwd_host(q, k, v, o, lse, B, H, T, d, int(bool(causal)), float(scale),
                             heads_per_chunk, ws, ws_bytes, stream)
