"""fp64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY.  This package is the reference the CUDA path is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import it; the library in
``exact_attention_tmem_gb300`` never does, and the two share no code.

The arithmetic lives in ``fa_oracle.c`` (plain C, OpenMP over rows/heads); each
function there cites the page and section it follows.  This module only builds
that file with gcc and marshals numpy arrays through ctypes.

Every function takes float64 arrays shaped [B, H, N, d] (already rounded to the
values the GPU receives) and returns float64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libfa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` (default fa_oracle.c) with gcc and OpenMP into ``out``."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, t=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(t))


def _shape4(*arrays):
    shape = arrays[0].shape
    if len(shape) != 4:
        raise ValueError("expected [B, H, N, d] arrays")
    for a in arrays[1:]:
        if a.shape != shape:
            raise ValueError("q, k, v (and dO) must share one [B, H, N, d] shape")
    return shape


class Oracle:
    """ctypes front end of one compiled copy of the oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
        lib.oracle_fwd_rows.argtypes = [dp, dp, dp, L, L, L, D, I, lp, L, dp, dp]
        lib.oracle_fwd_rows.restype = I
        lib.oracle_fwd.argtypes = [dp, dp, dp, L, L, L, D, I, dp, dp]
        lib.oracle_fwd.restype = I
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, L, L, L, D, I, dp, dp, dp]
        lib.oracle_bwd.restype = I
        lib.oracle_bwd_rows.argtypes = [dp, dp, dp, dp, L, L, L, D, I, lp, L, dp, dp, dp]
        lib.oracle_bwd_rows.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        self._lib = lib

    def num_threads(self) -> int:
        """OpenMP threads the oracle runs with."""
        return int(self._lib.oracle_num_threads())

    def attention_fwd(self, q, k, v, scale: float, causal: bool):
        """O = softmax(scale * Q K^T [masked]) V and L = logsumexp per row (natural log).

        Returns (O [B,H,N,d], L [B,H,N]) in float64.
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, d = _shape4(q, k, v)
        o = np.empty((B, H, N, d))
        lse = np.empty((B, H, N))
        rc = self._lib.oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B * H, N, d, float(scale),
                                  int(bool(causal)), _ptr(o), _ptr(lse))
        if rc:
            raise RuntimeError(f"oracle_fwd failed ({rc})")
        return o, lse

    def attention_fwd_rows(self, q, k, v, scale: float, causal: bool, rows):
        """Forward for the listed query rows of every head.

        rows: 1-D integer array of query indices.  Returns (O [B,H,R,d], L [B,H,R]).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, H, N, d = _shape4(q, k, v)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
        o = np.empty((B, H, R, d))
        lse = np.empty((B, H, R))
        rc = self._lib.oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B * H, N, d, float(scale),
                                       int(bool(causal)), _ptr(rows, ctypes.c_long), R,
                                       _ptr(o), _ptr(lse))
        if rc:
            raise RuntimeError(f"oracle_fwd_rows failed ({rc})")
        return o, lse

    def attention_bwd(self, q, k, v, dout, scale: float, causal: bool):
        """Gradients of sum(O * dO) w.r.t. Q, K, V.  Returns (dQ, dK, dV) in float64."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, N, d = _shape4(q, k, v, dout)
        dq = np.empty((B, H, N, d))
        dk = np.empty((B, H, N, d))
        dv = np.empty((B, H, N, d))
        rc = self._lib.oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B * H, N, d,
                                  float(scale), int(bool(causal)), _ptr(dq), _ptr(dk),
                                  _ptr(dv))
        if rc:
            raise RuntimeError(f"oracle_bwd failed ({rc})")
        return dq, dk, dv

    def attention_bwd_rows(self, q, k, v, dout, scale: float, causal: bool, rows):
        """Backward restricted to the listed query rows of every head.

        Returns (dQ of those rows [B,H,R,d], and the contributions of exactly those
        rows to dK and dV [B,H,N,d]).  With every row listed this is attention_bwd.
        """
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        B, H, N, d = _shape4(q, k, v, dout)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        R = rows.shape[0]
        dq = np.empty((B, H, R, d))
        dk = np.empty((B, H, N, d))
        dv = np.empty((B, H, N, d))
        rc = self._lib.oracle_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B * H, N, d,
                                       float(scale), int(bool(causal)),
                                       _ptr(rows, ctypes.c_long), R, _ptr(dq), _ptr(dk), _ptr(dv))
        if rc:
            raise RuntimeError(f"oracle_bwd_rows failed ({rc})")
        return dq, dk, dv


def default() -> Oracle:
    """The oracle built from fa_oracle.c (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
    return _lib


def num_threads() -> int:
    return default().num_threads()


def attention_fwd(q, k, v, scale: float, causal: bool):
    return default().attention_fwd(q, k, v, scale, causal)


def attention_fwd_rows(q, k, v, scale: float, causal: bool, rows):
    return default().attention_fwd_rows(q, k, v, scale, causal, rows)


def attention_bwd(q, k, v, dout, scale: float, causal: bool):
    return default().attention_bwd(q, k, v, dout, scale, causal)


def attention_bwd_rows(q, k, v, dout, scale: float, causal: bool, rows):
    return default().attention_bwd_rows(q, k, v, dout, scale, causal, rows)
