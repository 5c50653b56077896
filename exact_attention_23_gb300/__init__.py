"""Exact attention for GB300 (sm_103a).

``fwd(q, k, v, causal)`` returns ``(o, lse)`` for contiguous bf16 CUDA tensors of shape
[B, H, T, d] (d = 64 or 128): o = softmax(scale·QKᵀ [+causal mask])·V in bf16 and the
per-row natural-log logsumexp in fp32. ``fwd_kv`` attends Tq queries to Tk ≥ Tq keys
(bottom-right causal; key range split over CTAs when that fills the GPU), and
``fwd_block_sparse`` skips 128×128 blocks switched off by a block mask.
``bwd(q, k, v, o, lse, do, causal)`` returns the gradients (dq, dk, dv) (d = 64 or 128).
The work is done by the CUDA kernels of ``libfa.so`` through its C ABI (include/fa.h);
this module only allocates outputs and workspace with PyTorch and passes pointers and the
current stream.
"""

from __future__ import annotations

import math

from ._binding import (  # noqa: F401
    EXPORTS,
    FA_ERR_INVALID_ARG,
    FA_ERR_LAUNCH,
    FA_ERR_MISALIGNED,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED_DEVICE,
    FA_FLAG_TEST_STARVE_Q,
    FA_FLAG_TEST_STARVE_LATER_Q,
    FA_FLAG_CTA_PAIR,
    FA_OK,
    FAError,
    fa_bwd,
    fa_bwd_ex,
    fa_bwd_workspace_size,
    fa_fwd,
    fa_fwd_block_sparse,
    fa_fwd_ex,
    fa_fwd_fp8,
    fa_fwd_host,
    fa_fwd_host_workspace_size,
    fa_fwd_kv,
    fa_fwd_kv_workspace_size,
    lib,
    strerror,
    version,
)


def _check(t, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, T, d] tensor")


def fwd(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None,
        status=None, timeout_ns: int = 0, flags: int = 0):
    """Attention forward through libfa.so on the current CUDA stream.

    Returns (o, lse). ``out``/``lse`` may be given to reuse buffers. ``status``, an
    optional int32 CUDA tensor of one element, receives FA_ERR_TIMEOUT if an internal
    wait of the kernel ever gives up; ``timeout_ns`` bounds those waits (0: 2 s).
    ``flags`` is 0 except in tests of that path: FA_FLAG_TEST_STARVE_Q withholds every
    query-tile load, FA_FLAG_TEST_STARVE_LATER_Q those after each CTA's first unit; and
    FA_FLAG_CTA_PAIR (d = 64) runs the forward on CTA pairs sharing each tensor-core product
    (same results, slower on GB300 than the default).
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must have the same shape")
    B, H, T, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check(out, "out")
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    st_ptr = None if status is None else status.data_ptr()
    with torch.cuda.device(q.device):
        rc = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr(), B, H, T, d, causal, scale, st_ptr, timeout_ns, flags,
                       stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd")
    return out, lse


def fwd_host(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None,
             heads_per_chunk: int = 0, workspace=None, device=None, synchronize: bool = True):
    """Forward over host tensors (CPU bf16 [B, H, T, d], contiguous; page-locked for
    overlapped copies) through fa_fwd_host on ``device``'s current stream. Outputs are host
    tensors (page-locked when not given). With ``synchronize`` the stream is synchronised
    before returning; otherwise the caller must do so before reading them."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 \
                or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host bf16 [B, H, T, d] tensor")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must have the same shape")
    B, H, T, d = q.shape
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, pin_memory=True)
    with torch.cuda.device(dev):
        if workspace is None:
            need = fa_fwd_host_workspace_size(B, H, T, d, heads_per_chunk)
            if need == 0:
                raise FAError(FA_ERR_INVALID_ARG, "fa_fwd_host_workspace_size")
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        s = torch.cuda.current_stream(dev)
        rc = fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr(), B, H, T, d, causal, scale, heads_per_chunk,
                         workspace.data_ptr(), workspace.numel(), s.cuda_stream)
        if rc != FA_OK:
            raise FAError(rc, "fa_fwd_host")
        if synchronize:
            s.synchronize()
    return out, lse


def fwd_fp8(q8, q_scale: float, k8, k_scale: float, v, causal: bool = True,
            scale: float | None = None, out=None, lse=None):
    """Forward with e4m3 query/key codes (CUDA uint8 tensors [B, H, T, d]) and their
    per-tensor scales, bf16 v, through fa_fwd_fp8. Returns (o, lse)."""
    import torch
    for t, n in ((q8, "q8"), (k8, "k8")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.uint8 \
                or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CUDA uint8 [B, H, T, d] tensor")
    _check(v, "v")
    if q8.shape != k8.shape or q8.shape != v.shape:
        raise ValueError("q8, k8 and v must have the same shape")
    B, H, T, d = v.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(v) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=v.device)
    stream = torch.cuda.current_stream(v.device).cuda_stream
    with torch.cuda.device(v.device):
        rc = fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr(), q_scale, k_scale, B, H, T, d, causal, scale, stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_fp8")
    return out, lse


def fwd_kv(q, k, v, causal: bool = True, scale: float | None = None, n_splits: int = 0,
           out=None, lse=None, workspace=None):
    """Queries q [B, H, Tq, d] against keys/values k, v [B, H, Tk, d] through fa_fwd_kv.

    causal aligns bottom-right (query i sees key j iff j ≤ i + Tk − Tq; needs Tq ≤ Tk).
    n_splits = 0 lets the library choose how many key ranges to spread over CTAs; the
    workspace for the partial results is allocated here unless one is passed.
    Returns (o, lse); a row that sees no key has o = 0 and lse = −inf.
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B, H, Tq, d] and k, v [B, H, Tk, d]")
    B, H, Tq, d = q.shape
    Tk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, Tq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        need = fa_fwd_kv_workspace_size(B, H, Tq, Tk, d, n_splits)
        if need == 0:
            raise FAError(FA_ERR_INVALID_ARG, "fa_fwd_kv_workspace_size")
        if workspace is None and need > 1:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_ptr = None if workspace is None else workspace.data_ptr()
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        stream = torch.cuda.current_stream(q.device).cuda_stream
        rc = fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, Tq, Tk, d, causal, scale, n_splits, ws_ptr, ws_bytes, stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_kv")
    return out, lse


def fwd_block_sparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None,
                     out=None, lse=None):
    """Self-attention with 128×128 blocks switched off by ``block_mask`` (a CUDA uint8
    tensor [ceil(T/128), ceil(T/128)] shared by all heads, or [B·H, ...] per head;
    nonzero = compute), through fa_fwd_block_sparse. Returns (o, lse); a row that sees
    no key has o = 0 and lse = −inf."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must have the same shape")
    B, H, T, d = q.shape
    nb = q_tiles(T)
    if (not isinstance(block_mask, torch.Tensor) or not block_mask.is_cuda
            or block_mask.dtype != torch.uint8 or not block_mask.is_contiguous()):
        raise ValueError("block_mask must be a contiguous CUDA uint8 tensor")
    if tuple(block_mask.shape[-2:]) != (nb, nb) or block_mask.dim() not in (2, 3):
        raise ValueError(f"block_mask must be [{nb}, {nb}] or [B*H, {nb}, {nb}]")
    mask_heads = 1 if block_mask.dim() == 2 else block_mask.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        rc = fa_fwd_block_sparse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), block_mask.data_ptr(), mask_heads, B, H, T, d,
                                 causal, scale, stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_block_sparse")
    return out, lse


def bwd_workspace(B: int, H: int, T: int, d: int, device=None):
    """A uint8 CUDA tensor large enough to serve as fa_bwd's workspace (torch allocations
    are 256-byte aligned)."""
    import torch
    n = fa_bwd_workspace_size(B, H, T, d)
    if n == 0:
        raise FAError(FA_ERR_INVALID_ARG, "fa_bwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def bwd(q, k, v, o, lse, do, causal: bool = True, scale: float | None = None, dq=None,
        dk=None, dv=None, workspace=None, status=None, timeout_ns: int = 0, flags: int = 0):
    """Attention backward through libfa.so on the current CUDA stream.

    ``o`` and ``lse`` are the outputs of ``fwd`` for the same q, k, v, causal and scale;
    ``do`` is the gradient of the loss with respect to o. Returns (dq, dk, dv).
    ``workspace`` (see ``bwd_workspace``) may be passed to reuse it between calls.
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _check(t, n)
    if not (q.shape == k.shape == v.shape == o.shape == do.shape):
        raise ValueError("q, k, v, o and do must have the same shape")
    B, H, T, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, T] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n)
    if workspace is None:
        workspace = bwd_workspace(B, H, T, d, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    st_ptr = None if status is None else status.data_ptr()
    with torch.cuda.device(q.device):
        rc = fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                       B, H, T, d, causal, scale, st_ptr, timeout_ns, flags, stream)
    if rc != FA_OK:
        raise FAError(rc, "fa_bwd")
    return dq, dk, dv


def bwd_flops(B: int, H: int, T: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of one backward: five T×T×d products (S, dP, dV, dK, dQ), i.e.
    2.5 × the forward's count, halved when causal."""
    return 2.5 * flops(B, H, T, d, causal)


def flops(B: int, H: int, T: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of one forward: 4·B·H·T²·d (two T×T×d products), halved when
    causal (the convention the throughput figures are quoted in)."""
    f = 4.0 * B * H * T * T * d
    return f / 2.0 if causal else f


def hbm_bytes(B: int, H: int, T: int, d: int) -> float:
    """Algorithmic HBM bytes of one forward: read q, k, v once, write o (bf16) and lse (fp32)."""
    return B * H * T * (4.0 * d * 2 + 4.0)


def q_tiles(T: int, rows: int = 128) -> int:
    """Query-row tiles of ``rows`` rows covering a sequence of length T."""
    return -(-T // rows)
