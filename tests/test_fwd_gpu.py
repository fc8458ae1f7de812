"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16/fp32 inputs, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tmem_gb300 import inputs
from gpu_helpers import (assert_fwd_close, gpu_fwd, oracle_fwd, to_dev, max_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


# shapes spanning several tiles and ragged tails; N=1 and N < one tile included
SMALL = [
    (1, 1, 1, 64), (1, 2, 1, 128), (1, 1, 17, 64), (2, 1, 17, 128), (1, 2, 127, 64),
    (1, 1, 128, 128), (1, 2, 129, 64), (2, 2, 255, 128), (1, 3, 256, 64), (1, 1, 257, 128),
    (2, 3, 300, 64), (1, 2, 300, 128), (1, 2, 513, 128), (2, 2, 1000, 64), (1, 1, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SMALL)
def test_fwd_small_shapes(B, H, N, d, causal):
    q, k, v = inputs.random_inputs(B, H, N, d, seed=B * 1000 + H * 100 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal)
    o_ref, l_ref = oracle_fwd(q, k, v, causal, scale)
    assert_fwd_close(o, lse, o_ref, l_ref, f"B={B} H={H} N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row0_is_v0_exactly(d):
    """Query 0 sees only key 0 under the causal mask: O_0 = V_0 bit for bit
    (P_00 = 2^0 = 1 and l = 1), and L_0 = scale * q_0.k_0."""
    q, k, v = inputs.random_inputs(2, 2, 300, d, seed=77)
    qd, kd, vd = to_dev(q, k, v)
    import exact_attention_tmem_gb300 as fa
    o, lse = fa.fwd(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, 0].cpu(), v[:, :, 0])
    want = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1) / math.sqrt(d)
    assert float((lse[:, :, 0].cpu().double() - want).abs().max()) < 1e-4


@pytest.mark.parametrize("causal", [False, True])
def test_large_scores_exercise_rescaling(causal):
    """Scores with a spread of hundreds of units force the running max to move many
    times (the lazy rescale path), and late keys dominate some rows."""
    B, H, N, d = 1, 2, 700, 128
    q, k, v = inputs.random_inputs(B, H, N, d, seed=5)
    ramp = torch.linspace(0.2, 6.0, N).view(1, 1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q = (q.float() * 3.0).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal)
    o_ref, l_ref = oracle_fwd(q, k, v, causal, scale)
    assert_fwd_close(o, lse, o_ref, l_ref, f"large scores causal={causal}")


def test_spiky_keys_small():
    """The long-context recipe (1% of key rows scaled by 8) at a size the oracle
    checks in full."""
    shape = (1, 4, 1536, 128)
    q = inputs.normal(shape, 91)
    k = inputs.normal(shape, 92, spiky_rows_fraction=0.01)
    v = inputs.normal(shape, 93)
    o, lse = gpu_fwd(q, k, v, True)
    o_ref, l_ref = oracle_fwd(q, k, v, True, 1.0 / math.sqrt(128))
    assert_fwd_close(o, lse, o_ref, l_ref, "spiky keys")


@pytest.mark.parametrize("scale", [0.01, 0.5, 2.0])
def test_other_scales(scale):
    q, k, v = inputs.random_inputs(1, 2, 384, 64, seed=31)
    o, lse = gpu_fwd(q, k, v, True, scale=scale)
    o_ref, l_ref = oracle_fwd(q, k, v, True, scale)
    assert_fwd_close(o, lse, o_ref, l_ref, f"scale={scale}")


def test_deterministic_and_no_out_of_bounds_writes():
    """Two runs give identical bits; sentinel padding around o and lse is untouched."""
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 2, 3, 300, 128
    q, k, v = to_dev(*inputs.random_inputs(B, H, N, d, seed=3))
    n_o, n_l, pad = B * H * N * d, B * H * N, 4096
    o_buf = torch.full((n_o + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((n_l + pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[:n_o].view(B, H, N, d)
    lse = l_buf[:n_l].view(B, H, N)
    fa.fwd(q, k, v, causal=True, out=o, lse=lse)
    first = (o.clone(), lse.clone())
    fa.fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(first[0], o) and torch.equal(first[1], lse)
    assert bool((o_buf[n_o:] == 7.0).all()) and bool((l_buf[n_l:] == 7.0).all())
    assert bool(torch.isfinite(o.float()).all()) and bool(torch.isfinite(lse).all())


# ----------------------------------------------------------------- the five workloads

def test_workload1_f32_full():
    """fp32 inputs and outputs, B=1 H=1 N=256 d=64, non-causal: checked in full."""
    w = inputs.WORKLOADS[1]
    q, k, v = inputs.workload_inputs(1)
    o, lse = gpu_fwd(q, k, v, False)
    o_ref, l_ref = oracle_fwd(q, k, v, False, w.scale)
    assert_fwd_close(o, lse, o_ref, l_ref, "workload 1 (f32)")


@pytest.mark.parametrize("causal", [False, True])
def test_workload2_full(causal):
    """B=4 H=16 N=2048 d=64 bf16, both masks: every output checked."""
    w = inputs.WORKLOADS[2]
    q, k, v = inputs.workload_inputs(2)
    o, lse = gpu_fwd(q, k, v, causal)
    o_ref, l_ref = oracle_fwd(q, k, v, causal, w.scale)
    assert_fwd_close(o, lse, o_ref, l_ref, f"workload 2 causal={causal}")


def _sampled_check(wid, causal, rows_per_head=256, full_heads=()):
    w = inputs.WORKLOADS[wid]
    q, k, v = inputs.workload_inputs(wid)
    o, lse = gpu_fwd(q, k, v, causal)
    rows = inputs.sample_rows(w.N, rows_per_head, seed=wid)
    q64, k64, v64 = inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v)
    o_ref, l_ref = oracle.attention_fwd_rows(q64, k64, v64, w.scale, causal, rows)
    assert_fwd_close(o[:, :, rows], lse[:, :, rows], o_ref, l_ref, f"workload {wid} sampled rows")
    for (b, h) in full_heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_h, l_h = oracle.attention_fwd(q64[sl], k64[sl], v64[sl], w.scale, causal)
        assert_fwd_close(o[sl], lse[sl], o_h, l_h, f"workload {wid} head ({b},{h})")


@pytest.mark.slow
def test_workload3_sampled():
    """B=2 H=32 N=8192 d=128 causal: 256 sampled rows of every head, two heads in full."""
    _sampled_check(3, True, 256, full_heads=((0, 0), (1, 31)))


@pytest.mark.slow
def test_workload4_forward_sampled():
    """B=8 H=16 N=4096 d=128 causal forward: 256 sampled rows of every head."""
    _sampled_check(4, True, 256, full_heads=((7, 15),))


@pytest.mark.slow
def test_workload5_sampled():
    """B=1 H=8 N=131072 d=128 causal, spiky keys: 256 sampled query rows per head."""
    _sampled_check(5, True, 256)
