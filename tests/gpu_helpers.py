"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs, run the fp64 oracle on the same (rounded) values, compare.

Tolerances (bf16 storage, fp32 accumulation), from the workload specification:
max |dO| <= 2e-2 on O, max |dL| <= 5e-3 on the logsumexp, and for each gradient
tensor max |error| <= 5e-2 * max |oracle gradient|.  Where the exact gradient is
identically zero (N = 1: dQ = dK = 0, since P = 1 and dS = dP - D = 0) a relative
bound would reject fp32 rounding noise (~1e-7), so there, and only there, the bound
is the absolute 1e-4.
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


def grad_bound(g_ref):
    """The gradient tolerance for an oracle gradient tensor: 5e-2 * max |g_ref|, or the
    absolute 1e-4 when g_ref is identically zero."""
    scale = float(np.max(np.abs(g_ref))) if np.size(g_ref) else 0.0
    return TOL_GRAD_REL * scale if scale > 0.0 else TOL_GRAD_ABS


def assert_grad_close(g, g_ref, name, what=""):
    scale = float(np.max(np.abs(g_ref))) if np.size(g_ref) else 0.0
    bound = grad_bound(g_ref)
    e = max_err(g, g_ref)
    assert e <= bound, f"{what}: {name} max error {e:.3e} > {bound:.3e} (max |oracle| = {scale:.3e})"
    return e / max(scale, 1e-30)
