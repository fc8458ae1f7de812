"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, run the fp64 oracle on the same (rounded) values, compare.

Tolerances (bf16 storage, fp32 accumulation), from the workload specification:
max |dO| <= 2e-2 on O, max |dL| <= 5e-3 on the logsumexp, and for each gradient
tensor max |error| <= 5e-2 * max |oracle gradient| + 1e-4.  The absolute 1e-4 term
only matters where the exact gradient vanishes identically (N = 1: dQ = dK = 0),
where the relative bound alone would reject fp32 rounding noise (~1e-7).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from exact_attention_tmem_gb300 import inputs

TOL_O = 2e-2
TOL_L = 5e-3
TOL_GRAD_REL = 5e-2
TOL_GRAD_ABS = 1e-4


def to_dev(*ts):
    return [t.to("cuda", non_blocking=False) for t in ts]


def gpu_fwd(q, k, v, causal, scale=None):
    import exact_attention_tmem_gb300 as fa
    qd, kd, vd = to_dev(q, k, v)
    o, lse = fa.fwd(qd, kd, vd, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def oracle_fwd(q, k, v, causal, scale):
    return oracle.attention_fwd(inputs.as_f64(q), inputs.as_f64(k), inputs.as_f64(v), scale, causal)


def max_err(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.size == 0:
        return 0.0
    if not np.all(np.isfinite(a)):
        return math.inf
    return float(np.max(np.abs(a - b)))


def assert_fwd_close(o, lse, o_ref, lse_ref, what=""):
    eo, el = max_err(o, o_ref), max_err(lse, lse_ref)
    assert eo <= TOL_O, f"{what}: max|dO| = {eo:.3e} > {TOL_O}"
    assert el <= TOL_L, f"{what}: max|dL| = {el:.3e} > {TOL_L}"
    return eo, el


def assert_grad_close(g, g_ref, name, what=""):
    scale = float(np.max(np.abs(g_ref))) if g_ref.size else 0.0
    e = max_err(g, g_ref)
    assert e <= TOL_GRAD_REL * scale + TOL_GRAD_ABS, \
        f"{what}: {name} max error {e:.3e} > {TOL_GRAD_REL} * {scale:.3e} + {TOL_GRAD_ABS}"
    return e / max(scale, 1e-30)
