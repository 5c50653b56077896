"""fa_bwd_noalloc (the backward with the library's fixed device reservation as workspace)
against fa_bwd with a caller workspace, through the C ABI. Named so that it is collected
after every other test file: it must pass on its own and after everything else ran."""

import numpy as np
import pytest

import exact_attention_23_gb300 as fa
from exact_attention_23_gb300 import _binding, inputs


def test_noalloc_rejects_sizes_beyond_the_reservation():
    # B·H = 12 at T = 10497 needs 12 · 10624 · 66 · 4 bytes > 32 MiB: rejected on the host,
    # before any device is touched (fake, never-dereferenced addresses).
    A = 0x7F0000000000
    assert fa.fa_bwd_workspace_size(1, 12, 10497, 64) > _binding.FA_BWD_NOALLOC_SCRATCH_BYTES
    assert fa.fa_bwd_workspace_size(1, 12, 10496, 64) <= _binding.FA_BWD_NOALLOC_SCRATCH_BYTES
    ptrs = [A + i * (1 << 32) for i in range(9)]
    assert _binding.fa_bwd_noalloc(*ptrs, 1, 12, 10497, 64, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert _binding.fa_bwd_noalloc(*ptrs, 1, 12, 128, 96, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert _binding.fa_bwd_noalloc(0, *ptrs[1:], 1, 12, 128, 64, 1, 0.125, None) == fa.FA_ERR_INVALID_ARG


# Head dim 128 takes 64-query tiles and a transposed dQ accumulator layout in the same
# reservation; B1 H4 T777 (ragged last tile) exercises that layout.
_WIDE_RAGGED = inputs.Workload("wide_ragged_t777", 1, 4, 777, 128, True, 11)


@pytest.mark.gpu
@pytest.mark.parametrize("name,causal", [("tiny_causal", True), ("ragged_t1000", True),
                                         ("ragged_t1000", False), ("wide_ragged_t777", True),
                                         ("wide_ragged_t777", False)])
def test_noalloc_matches_fa_bwd_twice_in_a_row(name, causal):
    import torch
    w = _WIDE_RAGGED if name == _WIDE_RAGGED.name else inputs.WORKLOADS[name]
    q, k, v = (t.cuda() for t in inputs.workload_qkv(w))
    do = inputs.workload_do(w).cuda()
    o, lse = fa.fwd(q, k, v, causal=causal)
    ref = fa.bwd(q, k, v, o, lse, do, causal=causal)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        rc = _binding.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                     dv.data_ptr(), w.B, w.H, w.T, w.d, causal, w.scale, stream)
        assert rc == fa.FA_OK, fa.strerror(rc)
        torch.cuda.synchronize()
        # dK and dV come from the same deterministic kernel: identical bits
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]), f"call {call}"
        # dQ is summed with atomic adds in an unspecified order: equal within rounding
        a = dq.float().cpu().numpy()
        b = ref[0].float().cpu().numpy()
        assert np.all(np.isfinite(a))
        assert np.abs(a - b).max() <= 2e-2 * np.abs(b).max(), f"call {call}"
