"""CUDA graph capture of the library's calls.

With caller-owned outputs and workspaces, fa_fwd, fa_bwd (both routes) and fa_decode
enqueue kernels only: no allocation, no host synchronisation.  So a step captured
into a CUDA graph (the backward's and the decoding call's kernels are chained with
programmatic dependent launch, which capture turns into programmatic graph edges)
replays with the results of eager calls on the same inputs: bit for bit, except dQ of
the single-pass backward, whose fp32 reductions are summed in a varying order.
"""
import math

import pytest
import torch

from exact_attention_tmem_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


def _capture(step):
    """Runs `step` once on a side stream (one-time library set-up happens outside the
    capture), then captures it into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


@pytest.mark.parametrize("deterministic", [False, True])
def test_fwd_bwd_graph_replay_matches_eager(deterministic):
    import exact_attention_tmem_gb300 as fa
    B, H, N, d = 1, 4, 1000, 128
    dev = torch.device("cuda")
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    size = (fa.bwd_deterministic_workspace_size if deterministic else fa.bwd_workspace_size)(B, H, N, d)
    ws = torch.empty(size, dtype=torch.uint8, device=dev)

    def load(seed):
        for t, s in zip((q, k, v, do), range(4)):
            t.copy_(inputs.normal((B, H, N, d), seed + s))

    def step():
        fa.fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse)
        fa.bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws,
               deterministic=deterministic)

    load(16100)
    g = _capture(step)
    for seed in (16200, 16300):
        load(seed)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for name, a, b in zip(("o", "lse", "dk", "dv"), (got[0], got[1], got[3], got[4]), (o, lse, dk, dv)):
            assert torch.equal(a, b), f"{name} differs between the replayed graph and eager calls"
        if deterministic:
            assert torch.equal(got[2], dq), "deterministic dq differs between graph and eager"
        else:
            err = float((got[2].float() - dq.float()).abs().max())
            assert err <= 2.0 ** -7 * float(dq.float().abs().max()), f"dq differs by {err:.3e}"


def test_decode_graph_replay_matches_eager():
    import exact_attention_tmem_gb300 as fa
    B, H, Hkv, Nk, d = 2, 16, 2, 3000, 128
    dev = torch.device("cuda")
    q = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    k = torch.empty((B, Hkv, Nk, d), dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.decode_workspace_size(B, H, Hkv, Nk, d), dtype=torch.uint8, device=dev)

    def load(seed):
        q.copy_(inputs.normal((B, H, d), seed))
        k.copy_(inputs.normal((B, Hkv, Nk, d), seed + 1))
        v.copy_(inputs.normal((B, Hkv, Nk, d), seed + 2))

    def step():
        fa.decode(q, k, v, out=o, lse=lse, workspace=ws)

    load(16400)
    g = _capture(step)
    for seed in (16500, 16600):
        load(seed)
        g.replay()
        torch.cuda.synchronize()
        got_o, got_l = o.clone(), lse.clone()
        step()
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        assert torch.equal(got_o, o) and torch.equal(got_l, lse)
