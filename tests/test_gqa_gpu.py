"""Grouped-query attention (several query heads share one key/value head): parity of
fa_fwd_gqa / fa_bwd_gqa with the oracle applied to the key/value heads repeated for
every query head ("FlashAttention" deep dive, "Implementation notes": several query
heads map to one key/value head and nothing else changes).  dK and dV of a key/value
head are the sums over the query heads that share it."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tmem_gb300 import inputs
from gpu_helpers import assert_fwd_close, assert_grad_close, to_dev

pytestmark = pytest.mark.gpu

CASES = [  # B, H, Hkv, N, d
    (2, 8, 2, 300, 128),
    (1, 4, 1, 257, 64),     # multi-query attention
    (1, 6, 3, 1000, 128),
    (2, 4, 4, 129, 64),     # group of one: plain multi-head attention
]


def _inputs(B, H, Hkv, N, d, seed):
    q = inputs.normal((B, H, N, d), seed)
    k = inputs.normal((B, Hkv, N, d), seed + 1)
    v = inputs.normal((B, Hkv, N, d), seed + 2)
    do = inputs.normal((B, H, N, d), seed + 3)
    return q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Hkv,N,d", CASES)
def test_gqa_forward_and_backward(B, H, Hkv, N, d, causal):
    import exact_attention_tmem_gb300 as fa
    fa.build()
    G = H // Hkv
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = _inputs(B, H, Hkv, N, d, seed=500 + B * 100 + H * 10 + Hkv + N)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape

    f = inputs.as_f64
    k_rep, v_rep = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    o_ref, l_ref = oracle.attention_fwd(f(q), f(k_rep), f(v_rep), scale, causal)
    what = f"B={B} H={H} Hkv={Hkv} N={N} d={d} causal={causal}"
    assert_fwd_close(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, l_ref, what)
    dq_ref, dk_rep, dv_rep = oracle.attention_bwd(f(q), f(k_rep), f(v_rep), f(do), scale, causal)
    dk_ref = dk_rep.reshape(B, Hkv, G, N, d).sum(axis=2)
    dv_ref = dv_rep.reshape(B, Hkv, G, N, d).sum(axis=2)
    for name, g, r in (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)):
        assert_grad_close(g.float().cpu().numpy().astype(np.float64), r, name, what)
