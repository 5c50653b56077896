"""GPU tests of fa_fwd_host (the forward over host-resident tensors, chunked over heads with
overlapped copies): its outputs are bit-identical to fa_fwd on the same values (each head is
attended by the same kernel with the same arithmetic, whatever the chunking), for several
chunk sizes, both memory kinds, both head dims, causal and not, a ragged length, and the
same workspace used twice in a row; and it matches the fp64 oracle within the forward's
tolerances."""

import numpy as np
import pytest

import oracle
from exact_attention_23_gb300 import inputs

pytestmark = pytest.mark.gpu


def _device_ref(q, k, v, causal):
    import torch
    import exact_attention_23_gb300 as fa
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B,H,T,d,causal,hpc,pinned", [
    (2, 6, 1000, 64, True, 1, True),
    (2, 6, 1000, 64, True, 5, True),     # chunks of 5, 5 and 2 heads
    (2, 6, 1000, 64, False, 0, True),    # automatic chunking
    (1, 7, 777, 128, True, 3, True),
    (1, 4, 2048, 128, False, 2, False),  # pageable host memory
    (1, 3, 1, 64, True, 1, True),        # one row per head
    (3, 2, 300, 64, True, 100, True),    # one chunk holds every head
])
def test_fwd_host_matches_device_forward(B, H, T, d, causal, hpc, pinned):
    import torch
    import exact_attention_23_gb300 as fa
    q, k, v = inputs.make_qkv(B, H, T, d, 800 + T + d)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = fa.fwd_host(q, k, v, causal=causal, heads_per_chunk=hpc)
    o_ref, lse_ref = _device_ref(q, k, v, causal)
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)


def test_fwd_host_reuses_its_workspace_and_matches_the_oracle():
    import torch
    import exact_attention_23_gb300 as fa
    B, H, T, d = 2, 4, 1000, 64
    need = fa.fa_fwd_host_workspace_size(B, H, T, d, 3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    runs = []
    for seed in (11, 12):
        q, k, v = (t.pin_memory() for t in inputs.make_qkv(B, H, T, d, seed))
        o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
        lse = torch.empty((B, H, T), dtype=torch.float32, pin_memory=True)
        # both calls enqueued before any synchronisation: the second waits for the first
        fa.fwd_host(q, k, v, causal=True, out=o, lse=lse, heads_per_chunk=3, workspace=ws,
                    synchronize=False)
        runs.append((q, k, v, o, lse))
    torch.cuda.synchronize()
    for q, k, v, o, lse in runs:
        o_ref, lse_ref = oracle.attention(*(inputs.to_f64_numpy(t) for t in (q, k, v)), True,
                                          d ** -0.5)
        err = np.abs(o.float().double().numpy() - o_ref)
        assert err.max() <= 2e-2 and err.mean() <= 1e-3
        assert np.abs(lse.double().numpy() - lse_ref).max() <= 1e-3
        o_dev, lse_dev = _device_ref(q, k, v, True)
        assert torch.equal(o, o_dev) and torch.equal(lse, lse_dev)
