"""Decoding parity: fa_decode (split keys, partial (m, l, acc) triples merged on the
device) against the fp64 decoding oracle on the same seeded bf16 inputs, across head
dims, grouped-query ratios, ragged and tiny key counts, chunk counts and peaked
scores; plus the full-size decode workload (sampled heads)."""
import math

import numpy as np
import pytest
import torch

from exact_attention_tmem_gb300 import inputs
from gpu_helpers import TOL_L, TOL_O, to_dev
from oracle import decode as odec

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


def _inputs(B, H, Hkv, Nk, d, seed):
    q = inputs.normal((B, H, d), seed)
    k = inputs.normal((B, Hkv, Nk, d), seed + 1)
    v = inputs.normal((B, Hkv, Nk, d), seed + 2)
    return q, k, v


def _check(q, k, v, scale, what, chunks=0):
    import exact_attention_tmem_gb300 as fa
    o, lse = fa.decode(*to_dev(q, k, v), scale=scale, num_chunks=chunks)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    f = inputs.as_f64
    O_ref, L_ref = odec.attention_decode(f(q), f(k), f(v), scale)
    eo = float(np.abs(o.float().cpu().numpy() - O_ref).max())
    el = float(np.abs(lse.cpu().numpy() - L_ref).max())
    assert eo <= TOL_O, f"{what}: max |dO| {eo:.3e}"
    assert el <= TOL_L, f"{what}: max |dL| {el:.3e}"
    return o, lse


CASES = [  # B, H, Hkv, Nk, d
    (1, 1, 1, 1, 64), (1, 2, 2, 1, 128), (2, 4, 4, 17, 128), (1, 8, 2, 63, 64), (2, 8, 1, 64, 128),
    (1, 4, 4, 65, 64), (2, 6, 2, 1000, 128), (1, 16, 2, 4097, 128), (3, 5, 5, 2500, 64),
    (1, 7, 1, 777, 128), (2, 32, 8, 8192, 128),
    # larger groups (tensor-core kernel): 3, 9, 12, 16 query heads per key/value head
    (2, 12, 4, 2048, 64), (1, 9, 1, 130, 128), (2, 24, 2, 1100, 128), (1, 16, 1, 300, 64), (1, 32, 2, 5000, 128),
    (1, 4, 1, 1, 128), (2, 4, 2, 65, 64), (1, 16, 1, 64, 128),   # one key, a ragged stage, one full stage
]


@pytest.mark.parametrize("B,H,Hkv,Nk,d", CASES)
def test_decode_matches_oracle(B, H, Hkv, Nk, d):
    q, k, v = _inputs(B, H, Hkv, Nk, d, seed=12000 + B * 1000 + H * 50 + Hkv * 7 + Nk + d)
    _check(q, k, v, 1.0 / math.sqrt(d), f"B={B} H={H} Hkv={Hkv} Nk={Nk} d={d}")


@pytest.mark.parametrize("chunks", [1, 2, 3, 7, 64, 1000])
def test_decode_chunk_counts(chunks):
    """Any number of chunks (clamped to whole 64-key stages) gives the same result."""
    B, H, Hkv, Nk, d = 2, 4, 2, 3000, 128
    q, k, v = _inputs(B, H, Hkv, Nk, d, seed=13000 + chunks)
    _check(q, k, v, 1.0 / math.sqrt(d), f"chunks={chunks}", chunks=chunks)


@pytest.mark.parametrize("Hkv,d", [(4, 64), (1, 128)])
def test_decode_most_chunks(Hkv, d):
    """The largest chunk count the workspace holds (256 chunks of one 64-key stage): every
    slot of the merge's per-chunk table is used."""
    B, H, Nk = 1, 4, 256 * 64
    q, k, v = _inputs(B, H, Hkv, Nk, d, seed=13500 + Hkv + d)
    _check(q, k, v, 1.0 / math.sqrt(d), f"256 chunks Hkv={Hkv} d={d}", chunks=256)


def test_decode_peaked_scores():
    """Scores spread over hundreds of units: the per-stage and cross-chunk rescales."""
    B, H, Hkv, Nk, d = 1, 4, 4, 5000, 128
    q, k, v = _inputs(B, H, Hkv, Nk, d, seed=14000)
    q = (q.float() * 4.0).to(torch.bfloat16)
    ramp = torch.linspace(0.1, 3.0, Nk).view(1, 1, Nk, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    _check(q, k, v, 1.0 / math.sqrt(d), "peaked", chunks=0)
    _check(q, k, v, 1.0 / math.sqrt(d), "peaked, 1 chunk", chunks=1)


def test_decode_is_the_last_row_of_causal_forward():
    """The decode of the last query row equals the forward kernel's last causal row."""
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 1, 4, 1000, 128
    q, k, v = to_dev(*inputs.random_inputs(B, H, N, d, seed=15000))
    o_f, l_f = fa.fwd(q, k, v, causal=True)
    o_d, l_d = fa.decode(q[:, :, -1].contiguous(), k, v)
    torch.cuda.synchronize()
    assert float((o_f[:, :, -1].float() - o_d.float()).abs().max()) <= TOL_O
    assert float((l_f[:, :, -1] - l_d).abs().max()) <= TOL_L


def test_decode_writes_nothing_past_its_outputs():
    import exact_attention_tmem_gb300 as fa
    B, H, Hkv, Nk, d = 2, 8, 2, 1500, 64
    q, k, v = to_dev(*_inputs(B, H, Hkv, Nk, d, seed=16000))
    pad = 512
    ob = torch.full((B * H * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    lb = torch.full((B * H + pad,), 7.0, dtype=torch.float32, device="cuda")
    fa.decode(q, k, v, out=ob[:B * H * d].view(B, H, d), lse=lb[:B * H].view(B, H))
    torch.cuda.synchronize()
    assert bool((ob[B * H * d:] == 7.0).all()) and bool((lb[B * H:] == 7.0).all())


@pytest.mark.slow
def test_decode_workload_sampled_heads():
    """The decode workload (B=8 H=32 Hkv=8 Nk=32768 d=128): the full problem on the GPU,
    eight seeded query heads checked against the oracle."""
    import exact_attention_tmem_gb300 as fa
    B, H, Hkv, Nk, d = 8, 32, 8, 32768, 128
    q, k, v = _inputs(B, H, Hkv, Nk, d, seed=17000)
    o, lse = fa.decode(*to_dev(q, k, v))
    torch.cuda.synchronize()
    rng = np.random.default_rng(17001)
    f = inputs.as_f64
    for b, h in zip(rng.integers(0, B, 8), rng.integers(0, H, 8)):
        kv = h // (H // Hkv)
        O_ref, L_ref = odec.attention_decode(f(q[b:b + 1, h:h + 1]), f(k[b:b + 1, kv:kv + 1]),
                                             f(v[b:b + 1, kv:kv + 1]), 1.0 / math.sqrt(d))
        assert float(np.abs(o[b, h].float().cpu().numpy() - O_ref[0, 0]).max()) <= TOL_O
        assert abs(float(lse[b, h]) - L_ref[0, 0]) <= TOL_L


def test_decode_back_to_back_calls_share_a_workspace():
    """Two decoding calls enqueued back to back with one workspace and different inputs:
    the second call's split kernel writes the triples the first call's merge kernel
    (a dependent launch) reads; stream order must keep them apart.  Each result equals
    the same call made alone, bit for bit."""
    import exact_attention_tmem_gb300 as fa
    B, H, Hkv, Nk, d = 2, 16, 2, 3000, 128
    a = to_dev(*_inputs(B, H, Hkv, Nk, d, 15100))
    b = to_dev(*_inputs(B, H, Hkv, Nk, d, 15200))
    ws = torch.empty(fa.decode_workspace_size(B, H, Hkv, Nk, d), dtype=torch.uint8, device="cuda")
    alone = []
    for t in (a, b):
        alone.append(fa.decode(*t, workspace=ws))
        torch.cuda.synchronize()
    together = [fa.decode(*t, workspace=ws) for t in (a, b)]
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for x, y in zip(alone, together):
        assert torch.equal(x[0], y[0]) and torch.equal(x[1], y[1])
