"""fa_fwd_bwd_host: the forward + backward step on host tensors, pipelined over chunks of
heads, against the same step on device tensors (fa_fwd then fa_bwd) and, on a small
case, against the fp64 oracle.

Every head is an independent problem and the kernels compute each head the same way
whatever the launch holds, so o, lse, dk and dv must equal the device path bit for bit;
dQ is summed with reductions whose order varies, so it is compared within a tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tmem_gb300 import inputs
from gpu_helpers import assert_fwd_close, assert_grad_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


def device_step(q, k, v, do, causal, scale):
    import exact_attention_tmem_gb300 as fa
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return tuple(t.cpu() for t in (o, lse, dq, dk, dv))


def host_step(q, k, v, do, causal, scale, chunk, pinned=True):
    import exact_attention_tmem_gb300 as fa
    if pinned:
        q, k, v, do = (t.pin_memory() for t in (q, k, v, do))
    out = fa.fwd_bwd_host(q, k, v, do, causal=causal, scale=scale, chunk_heads=chunk)
    torch.cuda.current_stream().synchronize()
    assert fa.device_status() == 0
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("chunk", [0, 1, 3, 100])
def test_host_step_matches_device_step(d, causal, chunk):
    B, H, N = 2, 5, 300          # 10 heads: chunks of 1, 3 (ragged: 3+3+3+1), all, auto
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=61, with_grad_out=True)
    scale = 1.0 / math.sqrt(d)
    ref = device_step(q, k, v, do, causal, scale)
    got = host_step(q, k, v, do, causal, scale, chunk)
    for name, g, r in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
        if name == "dq":
            assert float((g.float() - r.float()).abs().max()) <= 1e-2 * float(r.float().abs().max())
        else:
            assert torch.equal(g, r), name


@pytest.mark.parametrize("chunk", [0, 2])
def test_host_step_odd_head_count(chunk):
    """33 heads: the automatic chunk of ceil(33 / 8) = 5 heads leaves a last chunk of 3,
    chunks of 2 a last chunk of 1; with 11 or 17 chunks every slot of the ring is reused
    several times.  Each head is computed once, in some chunk."""
    B, H, N, d = 3, 11, 130, 64
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=65, with_grad_out=True)
    ref = device_step(q, k, v, do, True, 0.125)
    got = host_step(q, k, v, do, True, 0.125, chunk)
    for name, g, r in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
        if name == "dq":
            assert float((g.float() - r.float()).abs().max()) <= 1e-2 * float(r.float().abs().max())
        else:
            assert torch.equal(g, r), name


def test_host_step_pageable_memory():
    """Pageable host buffers are correct too (the copies just do not overlap)."""
    B, H, N, d = 1, 4, 200, 128
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=62, with_grad_out=True)
    ref = device_step(q, k, v, do, True, 0.1)
    got = host_step(q, k, v, do, True, 0.1, chunk=2, pinned=False)
    for name, g, r in zip(("o", "lse", "dq", "dk", "dv"), got, ref):
        if name == "dq":
            assert float((g.float() - r.float()).abs().max()) <= 1e-2 * float(r.float().abs().max())
        else:
            assert torch.equal(g, r), name


def test_host_step_against_oracle():
    B, H, N, d = 1, 3, 257, 64
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=63, with_grad_out=True)
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = host_step(q, k, v, do, True, scale, chunk=2)
    f = inputs.as_f64
    o_ref, l_ref = oracle.attention_fwd(f(q), f(k), f(v), scale, True)
    assert_fwd_close(o.double().numpy(), lse.double().numpy(), o_ref, l_ref, "host step")
    ref = oracle.attention_bwd(f(q), f(k), f(v), f(do), scale, True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(g.double().numpy(), r, name, "host step")


def test_host_step_waits_for_earlier_work_on_the_stream():
    """Inputs written by a device->host copy enqueued just before the call are the
    ones the step reads: the step's copies start after earlier work on the stream."""
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 1, 2, 256, 128
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=64, with_grad_out=True)
    ref = device_step(q, k, v, do, False, 0.1)
    qd = q.cuda()
    torch.cuda.synchronize()
    hq = torch.zeros_like(q).pin_memory()
    hk, hv, hdo = (t.pin_memory() for t in (k, v, do))
    big = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    big.fill_(1)                           # keep the stream busy for a while
    hq.copy_(qd, non_blocking=True)        # q arrives in host memory only after that
    out = fa.fwd_bwd_host(hq, hk, hv, hdo, causal=False, scale=0.1, chunk_heads=1)
    torch.cuda.current_stream().synchronize()
    for name, g, r in zip(("o", "lse", "dq", "dk", "dv"), out, ref):
        if name == "dq":
            assert float((g.float() - r.float()).abs().max()) <= 1e-2 * float(r.float().abs().max())
        else:
            assert torch.equal(g, r), name


@pytest.mark.slow
def test_host_step_benchmarked_shape_against_oracle():
    """The end-to-end call the benchmark times: B=2 H=32 N=8192 d=128 causal on host
    buffers in chunks of 4 heads; o and lse on three seeded heads in full and 256 sampled
    rows of every head, the gradients of the same three heads in full, against the oracle."""
    import bench
    w = inputs.WORKLOADS[3]
    q, k, v, do = inputs.workload_inputs(3, with_grad_out=True)
    o, lse, dq, dk, dv = host_step(q, k, v, do, True, w.scale, chunk=bench.E2E_CHUNK_HEADS)
    f = inputs.as_f64
    heads = [(0, 0), (1, 31), (1, 7)]
    sel_b = [b for b, _ in heads]
    sel_h = [h for _, h in heads]
    sub = lambda t: f(t)[sel_b, sel_h][None]
    o_ref, l_ref = oracle.attention_fwd(sub(q), sub(k), sub(v), w.scale, True)
    assert_fwd_close(o.double().numpy()[sel_b, sel_h][None], lse.double().numpy()[sel_b, sel_h][None],
                     o_ref, l_ref, f"host step, workload 3 heads {heads}")
    rows = inputs.sample_rows(w.N, 256, seed=3303)
    o_s, l_s = oracle.attention_fwd_rows(f(q), f(k), f(v), w.scale, True, rows)
    assert_fwd_close(o.double().numpy()[:, :, rows], lse.double().numpy()[:, :, rows], o_s, l_s,
                     "host step, workload 3 sampled rows")
    ref = oracle.attention_bwd(sub(q), sub(k), sub(v), sub(do), w.scale, True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(g.double().numpy()[sel_b, sel_h][None], r, name, f"host step, workload 3 heads {heads}")
