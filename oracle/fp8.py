"""Oracle for the FP8 forward with incoherent processing.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it; the CUDA
library never does, and the two share no code.

The pages say only that the low-precision mode of the third-generation kernel runs in
FP8 "with incoherent processing" ("FlashAttention" deep dive, section "How it works";
"FlashAttention Explained", section "Later versions": FP8 low-precision mode).  The
plainest reading, taken here and by the CUDA path:

* FP8 is the e4m3 format (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  largest finite value 448, no infinities), values rounded to nearest with ties to
  even and clamped to +-448 (``e4m3_round``);
* incoherent processing multiplies each row of Q and of K by the same orthogonal
  matrix M = diag(s) H / sqrt(d), with H the d x d Sylvester Hadamard matrix and s a
  vector of random signs drawn by the caller, so that Q M (K M)^T = Q K^T while
  outlier coordinates are spread over the row before rounding (``rotate`` computes it
  with the fast Walsh-Hadamard butterflies, stride 1, 2, 4, ... in fp32, the order the
  kernel uses, so that both sides round the same fp32 values);
* each (batch, head) slice of Q, K and V gets one scale: descale = amax / 448 and
  codes = e4m3(x * (448 / amax)) with the two fp32 operations rounded as written
  (``quantize``);
* the attention itself is the plain definition applied to the dequantized values
  (``attention_dequantized``, fp64).

Arrays are numpy; shapes [B, H, N, d].
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_round(x):
    """Round float64 values (given exactly) to e4m3: nearest, ties to even, saturating
    at +-448.  Returns float64 values on the e4m3 grid (NaN stays NaN)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # spacing of the grid at |x|: 2^(e-3) for normals (e = floor(log2 |x|) >= -6),
    # 2^-9 in the subnormal range below 2^-6
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    step = np.exp2(e - 3.0)
    q = np.round(a / step) * step          # np.round: ties to even on the scaled grid
    q = np.minimum(q, E4M3_MAX)
    return np.where(np.isnan(x), np.nan, np.copysign(q, x))


def e4m3_code(v):
    """The 8-bit code of values already on the e4m3 grid (for bit-exact comparisons)."""
    v = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.uint8)
    sub = a < 2.0 ** -6
    code[sub] = np.round(a[sub] / 2.0 ** -9).astype(np.uint8)          # exponent field 0
    nz = ~sub
    e = np.floor(np.log2(a[nz])).astype(np.int64)
    m = np.round(a[nz] / np.exp2(e) * 8.0 - 8.0).astype(np.int64)       # 3 mantissa bits
    code[nz] = ((e + 7) << 3 | m).astype(np.uint8)
    return code | sign


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix: H[i, j] = (-1)^popcount(i & j), H H^T = d I."""
    i = np.arange(d)
    bits = np.bitwise_and.outer(i, i)
    pop = np.zeros_like(bits)
    while bits.any():
        pop += bits & 1
        bits >>= 1
    return np.where(pop % 2 == 0, 1.0, -1.0)


def rotate(x, signs):
    """Rows of x (float32 values) times diag(signs) H / sqrt(d), in fp32: the signs, then
    the butterflies (for stride 1, 2, 4, ...: x_i + x_{i+s} and x_i - x_{i+s}), then one
    multiply by the fp32 value of 1/sqrt(d)."""
    y = np.asarray(x, dtype=np.float32) * np.asarray(signs, dtype=np.float32)
    d = y.shape[-1]
    s = 1
    while s < d:
        y = y.reshape(y.shape[:-1] + (d // (2 * s), 2, s))
        a, b = y[..., 0, :], y[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(y.shape[:-3] + (d,))
        s *= 2
    return y * np.float32(1.0 / np.sqrt(d))


def quantize(x):
    """Per-(batch, head) e4m3 quantization of float32 values x [B, H, N, d]: returns
    (codes as e4m3-grid float64 values, descale [B, H] float32) with
    descale = amax / 448 and values = e4m3(x * (448 / amax)), both fp32 operations."""
    x = np.asarray(x, dtype=np.float32)
    amax = np.abs(x).max(axis=(2, 3)).astype(np.float32)
    amax = np.where(amax > 0, amax, np.float32(1.0)).astype(np.float32)   # an all-zero head
    inv = (np.float32(E4M3_MAX) / amax).astype(np.float32)
    scaled = (x * inv[:, :, None, None]).astype(np.float32)
    return e4m3_round(scaled.astype(np.float64)), (amax / np.float32(E4M3_MAX)).astype(np.float32)


def attention_dequantized(q8, k8, v8, dq, dk, dv, scale: float, causal: bool, oracle_fwd):
    """The plain attention (fp64, through the C oracle's forward) of the dequantized
    tensors q8 * dq, k8 * dk, v8 * dv (per-head scales).  Returns (O, L)."""
    f = lambda a, s: np.asarray(a, dtype=np.float64) * np.asarray(s, dtype=np.float64)[:, :, None, None]
    return oracle_fwd(f(q8, dq), f(k8, dk), f(v8, dv), scale, causal)
