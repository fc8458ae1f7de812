"""Pins for the FP8 oracle (oracle/fp8.py): the e4m3 rounding against its definition's
fixed points and against torch's float8_e4m3fn conversion (a library routine), the
code table, the Hadamard matrix, the butterfly rotation against the matrix product, the
invariance of Q K^T under the rotation, and the quantization's per-head scale."""
import math

import numpy as np
import pytest
import torch

from oracle import fp8


def test_e4m3_fixed_points():
    r = fp8.e4m3_round
    assert r(1.0) == 1.0 and r(448.0) == 448.0 and r(-448.0) == -448.0
    assert r(1.0625) == 1.0          # halfway between 1 and 1.125: ties to even
    assert r(1.1875) == 1.25         # halfway between 1.125 and 1.25: ties to even
    assert r(464.0) == 448.0         # halfway to the (missing) 480: even side is 448
    assert r(1e6) == 448.0 and r(-1e6) == -448.0   # saturating
    assert r(2.0 ** -9) == 2.0 ** -9                # smallest subnormal
    assert r(2.0 ** -10) == 0.0                     # halfway to 0: ties to even
    assert r(3 * 2.0 ** -10) == 2.0 ** -8
    assert np.isnan(r(np.nan))


def test_e4m3_matches_torch_within_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1e-1, 1, 10, 100)])
    x = x[np.abs(x) <= 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x.astype(np.float64)), ref.astype(np.float64))


def test_e4m3_code_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ok = ~np.isnan(vals) & ~((codes & 0x7F) == 0)       # skip NaNs and the two zeros
    np.testing.assert_array_equal(fp8.e4m3_code(vals[ok]), codes[ok])
    assert fp8.e4m3_code(np.array([0.0]))[0] == 0


@pytest.mark.parametrize("d", [2, 8, 64, 128])
def test_hadamard(d):
    H = fp8.hadamard(d)
    np.testing.assert_array_equal(H @ H.T, d * np.eye(d))
    np.testing.assert_array_equal(H, H.T)
    assert (np.abs(H) == 1).all()


def test_rotation_equals_matrix_product_and_preserves_scores():
    rng = np.random.default_rng(2)
    d = 128
    s = rng.choice([-1.0, 1.0], size=d)
    Q = rng.standard_normal((2, 3, 17, d)).astype(np.float32)
    K = rng.standard_normal((2, 3, 17, d)).astype(np.float32)
    M = np.diag(s) @ fp8.hadamard(d) / math.sqrt(d)
    np.testing.assert_allclose(fp8.rotate(Q, s), Q.astype(np.float64) @ M, atol=1e-5)
    np.testing.assert_allclose(M @ M.T, np.eye(d), atol=1e-12)
    Qr, Kr = fp8.rotate(Q, s).astype(np.float64), fp8.rotate(K, s).astype(np.float64)
    np.testing.assert_allclose(Qr @ np.swapaxes(Kr, -1, -2), Q.astype(np.float64) @ np.swapaxes(K, -1, -2),
                               atol=1e-4)


def test_rotation_spreads_an_outlier():
    d = 128
    x = np.zeros((1, 1, 1, d), dtype=np.float32)
    x[..., 5] = 100.0
    y = fp8.rotate(x, np.ones(d))
    np.testing.assert_allclose(np.abs(y), 100.0 / math.sqrt(d), rtol=1e-6)


def test_quantize_scale_and_range():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 2, 33, 16)).astype(np.float32)
    x[1, 0] *= 50
    vals, descale = fp8.quantize(x)
    amax = np.abs(x).max(axis=(2, 3))
    np.testing.assert_allclose(descale, amax / 448, rtol=1e-7)
    assert np.abs(vals).max() <= 448
    # the largest element of each head maps to (about) +-448
    for b in range(2):
        for h in range(2):
            assert abs(np.abs(vals[b, h]).max() - 448) <= 32
    # dequantized values are within half an e4m3 step (2^-4 relative) of the input
    deq = vals * descale[:, :, None, None]
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * descale[:, :, None, None])
    assert rel.max() <= 2.0 ** -4 + 1e-6
