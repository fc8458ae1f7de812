"""Backward parity: dQ, dK, dV from the CUDA path (through the C ABI) against the fp64
oracle on the same seeded bf16 inputs.  The GPU backward consumes the GPU forward's O
and logsumexp, as a user's training step would."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tmem_gb300 import inputs
from gpu_helpers import assert_grad_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


def gpu_fwd_bwd(q, k, v, do, causal, scale=None):
    import exact_attention_tmem_gb300 as fa
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return tuple(t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv))


def check_grads(q, k, v, do, causal, scale, what):
    got = gpu_fwd_bwd(q, k, v, do, causal, scale)
    f = inputs.as_f64
    ref = oracle.attention_bwd(f(q), f(k), f(v), f(do), scale, causal)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert_grad_close(g, r, name, what)


SMALL = [
    (1, 1, 1, 64), (1, 2, 1, 128), (1, 1, 17, 128), (2, 1, 17, 64), (1, 2, 128, 128),
    (1, 1, 129, 64), (2, 2, 255, 128), (1, 3, 256, 64), (2, 3, 300, 64), (1, 2, 300, 128),
    (1, 2, 513, 128), (1, 1, 1000, 64), (1, 1, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SMALL)
def test_bwd_small_shapes(B, H, N, d, causal):
    q, k, v, do = inputs.random_inputs(B, H, N, d, seed=B * 7000 + H * 300 + N + d, with_grad_out=True)
    check_grads(q, k, v, do, causal, 1.0 / math.sqrt(d), f"B={B} H={H} N={N} d={d} causal={causal}")


@pytest.mark.parametrize("scale", [0.05, 0.4])
def test_bwd_other_scales(scale):
    q, k, v, do = inputs.random_inputs(1, 2, 384, 128, seed=41, with_grad_out=True)
    check_grads(q, k, v, do, True, scale, f"scale={scale}")


def test_bwd_large_scores():
    """Peaked softmax rows (scores spread over hundreds of units)."""
    q, k, v, do = inputs.random_inputs(1, 2, 640, 128, seed=43, with_grad_out=True)
    q = (q.float() * 3.0).to(torch.bfloat16)
    ramp = torch.linspace(0.2, 5.0, 640).view(1, 1, 640, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    check_grads(q, k, v, do, True, 1.0 / math.sqrt(128), "large scores")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_dk_dv_deterministic_and_in_bounds(d):
    """dK and dV involve no atomics: two runs agree bit for bit; dQ is summed with
    reductions whose order varies, so only its last bits may differ.  Sentinel padding
    around every gradient buffer is untouched."""
    import exact_attention_tmem_gb300 as fa
    B, H, N = 2, 2, 300
    q, k, v, do = to_dev(*inputs.random_inputs(B, H, N, d, seed=45, with_grad_out=True))
    o, lse = fa.fwd(q, k, v, causal=True)
    n, pad = B * H * N * d, 2048
    bufs = [torch.full((n + pad,), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    grads = [b[:n].view(B, H, N, d) for b in bufs]
    fa.bwd(q, k, v, o, lse, do, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    first = [g.clone() for g in grads]
    fa.bwd(q, k, v, o, lse, do, causal=True, dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    assert torch.equal(first[1], grads[1]) and torch.equal(first[2], grads[2])
    assert float((first[0].float() - grads[0].float()).abs().max()) < 1e-2
    for b in bufs:
        assert bool((b[n:] == 3.0).all())
    for g in grads:
        assert bool(torch.isfinite(g.float()).all())


def test_bwd_workspace_contents_do_not_matter():
    """The workspace is scratch: garbage on entry gives the same gradients."""
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 1, 2, 257, 64
    q, k, v, do = to_dev(*inputs.random_inputs(B, H, N, d, seed=47, with_grad_out=True))
    o, lse = fa.fwd(q, k, v, causal=False)
    ws = torch.full((fa.bwd_workspace_size(B, H, N, d),), 0x7F, dtype=torch.uint8, device="cuda")
    g1 = fa.bwd(q, k, v, o, lse, do, causal=False, workspace=ws)
    ws.fill_(0xFF)
    g2 = fa.bwd(q, k, v, o, lse, do, causal=False, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert float((g1[0].float() - g2[0].float()).abs().max()) < 1e-2


@pytest.mark.slow
def test_workload4_backward_eight_heads():
    """B=8 H=16 N=4096 d=128 causal: the full problem on the GPU; eight seeded
    (batch, head) pairs checked in full against the oracle (dK and dV need every row)."""
    w = inputs.WORKLOADS[4]
    q, k, v, do = inputs.workload_inputs(4, with_grad_out=True)
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, True, w.scale)
    rng = np.random.default_rng(4004)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, w.B, 8), rng.integers(0, w.H, 8))]
    f = inputs.as_f64
    sel_b = [b for b, _ in heads]
    sel_h = [h for _, h in heads]
    sub = lambda t: f(t)[sel_b, sel_h][None]
    ref = oracle.attention_bwd(sub(q), sub(k), sub(v), sub(do), w.scale, True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(g[sel_b, sel_h][None], r, name, f"workload 4 heads {heads}")


@pytest.mark.slow
def test_default_bwd_benchmarked_shape():
    """B=2 H=32 N=8192 d=128 causal, the benchmarked problem, through fa_bwd (the
    single-pass route the benchmark times: dQ summed with bulk reductions); three seeded
    (batch, head) pairs checked in full against the oracle."""
    w = inputs.WORKLOADS[3]
    q, k, v, do = inputs.workload_inputs(3, with_grad_out=True)
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, True, w.scale)
    heads = [(0, 0), (1, 31), (1, 7)]
    sel_b = [b for b, _ in heads]
    sel_h = [h for _, h in heads]
    f = inputs.as_f64
    sub = lambda t: f(t)[sel_b, sel_h][None]
    ref = oracle.attention_bwd(sub(q), sub(k), sub(v), sub(do), w.scale, True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert_grad_close(g[sel_b, sel_h][None], r, name, f"workload 3 heads {heads}")


@pytest.mark.parametrize("deterministic", [False, True])
def test_bwd_back_to_back_calls_share_a_workspace(deterministic):
    """Two backward calls enqueued back to back on one stream with one workspace and
    different inputs.  The pre-processing of the second call may start as its
    predecessor's dependent launch; every call must still see only its own D, L and
    accumulator: each matches the same call made alone (dK and dV bit for bit)."""
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 1, 4, 1000, 128
    scale = 1.0 / math.sqrt(d)
    a = to_dev(*inputs.random_inputs(B, H, N, d, seed=4711, with_grad_out=True))
    b = to_dev(*inputs.random_inputs(B, H, N, d, seed=4712, with_grad_out=True))
    fo = [fa.fwd(t[0], t[1], t[2], causal=True, scale=scale) for t in (a, b)]
    size = (fa.bwd_deterministic_workspace_size if deterministic else fa.bwd_workspace_size)(B, H, N, d)
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    alone = []
    for t, (o, lse) in zip((a, b), fo):
        alone.append(fa.bwd(t[0], t[1], t[2], o, lse, t[3], causal=True, scale=scale, workspace=ws,
                            deterministic=deterministic))
        torch.cuda.synchronize()
    together = [fa.bwd(t[0], t[1], t[2], o, lse, t[3], causal=True, scale=scale, workspace=ws,
                       deterministic=deterministic) for t, (o, lse) in zip((a, b), fo)]
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for x, y in zip(alone, together):
        assert torch.equal(x[1], y[1]) and torch.equal(x[2], y[2])
        if deterministic:
            assert torch.equal(x[0], y[0])
        else:
            assert float((x[0].float() - y[0].float()).abs().max()) <= 1e-2 * float(x[0].float().abs().max())
