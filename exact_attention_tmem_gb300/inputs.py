"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it draws iid normal numbers with
numpy's PCG64 generator, optionally scales a seeded subset of key rows, and
rounds to the storage dtype.  The same tensors feed the CUDA path and, as their
exact float64 values, the CPU oracle.

Seeds follow one rule: ``seed = 1000 * workload_id + {q: 1, k: 2, v: 3, do: 4}``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_TENSOR_SEED = {"q": 1, "k": 2, "v": 3, "do": 4}


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, storage dtype, masks, and how it is checked."""
    wid: int
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str                      # "bf16" or "f32" storage for q, k, v, o
    causal: tuple                   # mask settings run on this workload
    backward: bool = False
    spiky_k_fraction: float = 0.0   # fraction of key rows per head scaled by spiky_k_factor
    spiky_k_factor: float = 8.0
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self, causal: bool) -> float:
        """4 N^2 d per head for the two forward contractions, halved when causal."""
        f = 4.0 * self.N * self.N * self.d * self.B * self.H
        return f / 2 if causal else f


WORKLOADS = {
    1: Workload(1, "fwd f32 B=1 H=1 N=256 d=64", 1, 1, 256, 64, "f32", (False,),
                note="fp32 inputs and outputs; the smallest case, checked in full"),
    2: Workload(2, "fwd bf16 B=4 H=16 N=2048 d=64", 4, 16, 2048, 64, "bf16", (False, True)),
    3: Workload(3, "fwd bf16 B=2 H=32 N=8192 d=128 causal", 2, 32, 8192, 128, "bf16", (True,)),
    4: Workload(4, "fwd+bwd bf16 B=8 H=16 N=4096 d=128 causal", 8, 16, 4096, 128, "bf16",
                (True,), backward=True),
    5: Workload(5, "fwd bf16 B=1 H=8 N=131072 d=128 causal, spiky K", 1, 8, 131072, 128,
                "bf16", (True,), spiky_k_fraction=0.01,
                note="1% of key rows per head scaled by 8 before rounding"),
}


def seed_for(wid: int, tensor: str) -> int:
    return 1000 * wid + _TENSOR_SEED[tensor]


def _torch_dtype(dtype: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def normal(shape, seed: int, dtype: str = "bf16", spiky_rows_fraction: float = 0.0,
           spiky_factor: float = 8.0) -> torch.Tensor:
    """iid N(0,1) in float64, optional row spikes, then rounded to ``dtype`` (CPU tensor).

    With ``spiky_rows_fraction`` > 0, floor(fraction * N) rows of every [N, d]
    slice (chosen by a seeded permutation) are multiplied by ``spiky_factor``
    before rounding.
    """
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=tuple(shape))
    if spiky_rows_fraction > 0.0:
        B, H, N = shape[0], shape[1], shape[2]
        n_spiky = int(math.floor(spiky_rows_fraction * N))
        sel = np.random.default_rng(seed + 500)
        for b in range(B):
            for h in range(H):
                rows = sel.permutation(N)[:n_spiky]
                x[b, h, rows, :] *= spiky_factor
    return torch.from_numpy(x).to(_torch_dtype(dtype))


def workload_inputs(wid: int, with_grad_out: bool = False, n_override: int | None = None):
    """q, k, v (and dO) CPU tensors for workload ``wid``.

    ``n_override`` replaces N (for scaled-down variants of a workload's recipe).
    """
    w = WORKLOADS[wid]
    N = n_override if n_override is not None else w.N
    shape = (w.B, w.H, N, w.d)
    q = normal(shape, seed_for(wid, "q"), w.dtype)
    k = normal(shape, seed_for(wid, "k"), w.dtype, w.spiky_k_fraction, w.spiky_k_factor)
    v = normal(shape, seed_for(wid, "v"), w.dtype)
    if not with_grad_out:
        return q, k, v
    do = normal(shape, seed_for(wid, "do"), w.dtype)
    return q, k, v, do


def random_inputs(B, H, N, d, seed: int, dtype: str = "bf16", with_grad_out: bool = False):
    """Seeded iid normal q, k, v (, dO) of an arbitrary shape (edge-case tests)."""
    shape = (B, H, N, d)
    out = [normal(shape, seed * 10 + i, dtype) for i in range(4 if with_grad_out else 3)]
    return tuple(out)


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a CPU tensor (what the oracle is given)."""
    return t.detach().to("cpu", torch.float64).numpy()


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct query rows: the first and last rows plus seeded random ones."""
    count = min(count, N)
    rng = np.random.default_rng(seed)
    fixed = {0, N - 1, min(N - 1, 127), min(N - 1, 128)}
    rest = rng.choice(N, size=count, replace=False)
    rows = sorted(fixed | set(int(r) for r in rest))
    return np.array(rows[:max(count, len(fixed))], dtype=np.int64)
