"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory
(for instance a plugin that a framework hands only its tensors, or a loop that must not
call cudaMalloc).  It uses a scratch array built into the library instead of a
caller-owned workspace; its results must match fa_bwd's.

This file is named so that pytest collects it last."""
import ctypes
import math

import pytest
import torch

from exact_attention_tmem_gb300 import _lib, inputs
from gpu_helpers import assert_grad_close, to_dev

pytestmark = pytest.mark.gpu


def _noalloc_bwd(q, k, v, o, lse, do, causal, scale):
    lib = _lib.load()
    B, H, N, d = q.shape
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                            ctypes.c_float(scale), int(causal), torch.cuda.current_stream().cuda_stream)
    _lib.check(st, "fa_bwd_noalloc")
    return dq, dk, dv


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_noalloc_backward_matches_fa_bwd_twice(d, causal):
    import exact_attention_tmem_gb300 as fa
    fa.build()
    B, H, N = 2, 3, 300
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = to_dev(*inputs.random_inputs(B, H, N, d, seed=909 + d, with_grad_out=True))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    ref = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)   # caller-owned workspace
    torch.cuda.synchronize()
    for call in range(2):                                          # two calls in a row
        got = _noalloc_bwd(q, k, v, o, lse, do, causal, scale)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_grad_close(g.float().cpu().numpy(), r.float().cpu().numpy(), name,
                              f"no-alloc call {call + 1}, d={d}, causal={causal}")


def test_noalloc_backward_near_the_scratch_limit():
    """A problem whose workspace fills the built-in array to within one 128-row tile
    (the per-row vectors sit past the dQ accumulator, at the top of the array): the
    results match fa_bwd with a caller-owned workspace."""
    import exact_attention_tmem_gb300 as fa
    fa.build()
    lib = _lib.load()
    B, H, d = 1, 4, 128
    limit = _lib.NOALLOC_SCRATCH_BYTES
    lo, hi = 1, 1 << 20
    while lo < hi:                      # the largest N whose workspace fits
        mid = (lo + hi + 1) // 2
        if lib.fa_bwd_workspace_size(B, H, mid, d) <= limit:
            lo = mid
        else:
            hi = mid - 1
    N = lo
    need = lib.fa_bwd_workspace_size(B, H, N, d)
    assert limit - 128 * (B * H) * (d * 4 + 8) < need <= limit
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = to_dev(*inputs.random_inputs(B, H, N, d, seed=919, with_grad_out=True))
    o, lse = fa.fwd(q, k, v, causal=True, scale=scale)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    for call in range(2):
        got = _noalloc_bwd(q, k, v, o, lse, do, True, scale)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2])
        assert_grad_close(got[0].float().cpu().numpy(), ref[0].float().cpu().numpy(), "dQ",
                          f"no-alloc near the limit (N={N}), call {call + 1}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    B, H, N, d = 8, 16, 4096, 128       # needs ~260 MB of scratch
    assert lib.fa_bwd_workspace_size(B, H, N, d) > _lib.NOALLOC_SCRATCH_BYTES
    fake = 0x10000                      # never dereferenced: rejected before any launch
    st = lib.fa_bwd_noalloc(*([fake] * 9), B, H, N, d, ctypes.c_float(0.1), 1, None)
    assert st == _lib.FA_ERR_WORKSPACE
