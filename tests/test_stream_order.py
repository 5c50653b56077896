"""Stream order under programmatic dependent launch. Every kernel of the library starts its
set-up before the previous kernel on the stream has finished and waits for it before
touching global memory. These tests enqueue chains in which each call consumes the result
of the kernel just before it, with no synchronisation in between, and check the results
are bit-identical to the same calls run one at a time with a synchronisation after each."""

import pytest

from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu


def _sync():
    import torch
    torch.cuda.synchronize()


def test_forward_consumes_the_kernel_just_before_it():
    """q, k, v produced by a PyTorch kernel on the same stream, attended at once; then the
    output fed straight back in as the next call's queries."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 2, 6, 2048, 64
    q0, k0, v0 = (t.cuda() for t in inputs.make_qkv(B, H, T, d, 41))

    def chain(sync_each):
        q = (q0.float() * 1.5).to(torch.bfloat16)   # a device kernel right before the call
        if sync_each:
            _sync()
        o1, l1 = fa.fwd(q, k0, v0, causal=True)
        if sync_each:
            _sync()
        o2, l2 = fa.fwd(o1, k0, v0, causal=False)  # consumes the previous forward's output
        if sync_each:
            _sync()
        return o1, l1, o2, l2

    got = chain(False)
    _sync()
    want = chain(True)
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_backward_then_forward_chain():
    """forward → backward (reads o and lse) → forward on the gradient dq, all enqueued
    back to back."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 1, 4, 1000, 64
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, T, d, 42))
    do = inputs.make_do(B, H, T, d, 42).cuda()

    def chain(sync_each):
        o, lse = fa.fwd(q, k, v, causal=True)
        if sync_each:
            _sync()
        dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=True)
        if sync_each:
            _sync()
        o3, l3 = fa.fwd(dq, dk, dv, causal=True)
        if sync_each:
            _sync()
        return o, lse, dq, dk, dv, o3, l3

    got = chain(False)
    _sync()
    want = chain(True)
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_decode_calls_back_to_back():
    """Decode with its key-range merge, called repeatedly on the same buffers (each call's
    split kernel overwrites the partials the previous call's merge reads), with a device
    kernel changing the query between calls."""
    import torch
    import exact_attention_23_gb300 as fa
    B, H, Tk, d = 2, 6, 4096, 64
    q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Tk, d, 43))
    q1 = q[:, :, -1:].contiguous()

    def chain(sync_each):
        outs = []
        qq = q1.clone()
        for _ in range(4):
            o, lse = fa.fwd_kv(qq, k, v, causal=True, n_splits=0)
            if sync_each:
                _sync()
            outs += [o, lse]
            qq = (o.float() + qq.float()).to(torch.bfloat16)  # depends on this call's output
            if sync_each:
                _sync()
        return outs

    got = chain(False)
    _sync()
    want = chain(True)
    for a, b in zip(got, want):
        assert torch.equal(a, b)
