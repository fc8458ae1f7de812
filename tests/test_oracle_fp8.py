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


# ---------------------------------------------------------------------------------------
# attention_dequantized: the per-head descales must reach the right tensor on the right
# axis.  Pinned by closed forms that hold whatever the codes are:
#   * V constant per head (codes 1, descale c_bh): every softmax row sums to one, so
#     O[b, h] = c_bh exactly;
#   * one key (N = 1): L[b, h, 0] = scale * (dq_bh q8 . dk_bh k8) = scale dq dk (q8 . k8)
#     and O = dv_bh v8[0];
#   * Q codes zero: every score is 0, so L = ln N and O = the mean of dv_bh v8 over keys;
#   * moving a factor between a code tensor and its descale changes nothing.
# Descales differ by orders of magnitude between heads and B != H, so a descale taken
# on the wrong axis, dk used for dq, or a scale dropped fails one of these.
# ---------------------------------------------------------------------------------------
import oracle  # noqa: E402


def _descales(rng, B, H):
    return (10.0 ** rng.uniform(-3, 1, size=(B, H))).astype(np.float32)


def _codes(rng, shape):
    return fp8.e4m3_round(rng.standard_normal(shape) * 40.0)


def test_dequantized_constant_v_gives_its_scale():
    rng = np.random.default_rng(11)
    B, H, N, d = 2, 3, 37, 16
    q8, k8 = _codes(rng, (B, H, N, d)), _codes(rng, (B, H, N, d))
    dq, dk, dv = _descales(rng, B, H), _descales(rng, B, H), _descales(rng, B, H)
    v8 = np.ones((B, H, N, d))
    for causal in (False, True):
        o, _ = fp8.attention_dequantized(q8, k8, v8, dq, dk, dv, 0.25, causal, oracle.attention_fwd)
        want = np.broadcast_to(dv.astype(np.float64)[:, :, None, None], o.shape)
        np.testing.assert_allclose(o, want, rtol=1e-13, atol=0)


def test_dequantized_one_key_closed_form():
    rng = np.random.default_rng(12)
    B, H, d = 3, 2, 32
    q8, k8, v8 = _codes(rng, (B, H, 1, d)), _codes(rng, (B, H, 1, d)), _codes(rng, (B, H, 1, d))
    dq, dk, dv = _descales(rng, B, H), _descales(rng, B, H), _descales(rng, B, H)
    scale = 0.125
    o, lse = fp8.attention_dequantized(q8, k8, v8, dq, dk, dv, scale, False, oracle.attention_fwd)
    for b in range(B):
        for h in range(H):
            dot = float(np.dot(q8[b, h, 0], k8[b, h, 0]))
            want_l = scale * float(dq[b, h]) * float(dk[b, h]) * dot
            assert abs(lse[b, h, 0] - want_l) <= 1e-12 * max(1.0, abs(want_l))
            np.testing.assert_allclose(o[b, h, 0], float(dv[b, h]) * v8[b, h, 0], rtol=1e-13, atol=0)


def test_dequantized_zero_queries_give_uniform_weights():
    rng = np.random.default_rng(13)
    B, H, N, d = 2, 3, 29, 16
    k8, v8 = _codes(rng, (B, H, N, d)), _codes(rng, (B, H, N, d))
    dq, dk, dv = _descales(rng, B, H), _descales(rng, B, H), _descales(rng, B, H)
    q8 = np.zeros((B, H, N, d))
    o, lse = fp8.attention_dequantized(q8, k8, v8, dq, dk, dv, 0.3, False, oracle.attention_fwd)
    np.testing.assert_allclose(lse, math.log(N), rtol=0, atol=1e-13)
    for b in range(B):
        for h in range(H):
            mean_v = float(dv[b, h]) * v8[b, h].mean(axis=0)
            np.testing.assert_allclose(o[b, h], np.broadcast_to(mean_v, (N, d)), rtol=1e-12, atol=1e-15)


def test_dequantized_factor_moves_between_codes_and_descale():
    rng = np.random.default_rng(14)
    B, H, N, d = 1, 2, 20, 16
    q8, k8, v8 = _codes(rng, (B, H, N, d)), _codes(rng, (B, H, N, d)), _codes(rng, (B, H, N, d))
    dq, dk, dv = _descales(rng, B, H), _descales(rng, B, H), _descales(rng, B, H)
    base = fp8.attention_dequantized(q8, k8, v8, dq, dk, dv, 0.2, True, oracle.attention_fwd)
    for which in range(3):
        codes, scales = [q8, k8, v8], [dq, dk, dv]
        codes[which] = codes[which] * 4.0
        scales[which] = (scales[which] / np.float32(4.0)).astype(np.float32)
        got = fp8.attention_dequantized(*codes, *scales, 0.2, True, oracle.attention_fwd)
        np.testing.assert_allclose(got[0], base[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(got[1], base[1], rtol=1e-12, atol=1e-12)


def _pins_pass(fn, monkeypatch):
    """Runs the pins above with fp8.attention_dequantized replaced by `fn`."""
    monkeypatch.setattr(fp8, "attention_dequantized", fn)
    try:
        test_dequantized_constant_v_gives_its_scale()
        test_dequantized_one_key_closed_form()
        test_dequantized_zero_queries_give_uniform_weights()
        test_dequantized_factor_moves_between_codes_and_descale()
    except AssertionError:
        return False
    return True


def _mutant(kind):
    def fn(q8, k8, v8, dq, dk, dv, scale, causal, oracle_fwd):
        def f(a, s):
            s = np.asarray(s, dtype=np.float64)
            if kind == "axis":     # descale indexed [h, b] instead of [b, h]
                s = s.T if s.shape[0] != s.shape[1] else s[::-1, ::-1]
                s = np.resize(s, (np.shape(a)[0], np.shape(a)[1]))
            return np.asarray(a, dtype=np.float64) * s[:, :, None, None]
        if kind == "dk_for_dq":
            dq = dk
        if kind == "no_dv":
            dv = np.ones_like(dv)
        if kind == "dv_for_dk":
            dk = dv
        return oracle_fwd(f(q8, dq), f(k8, dk), f(v8, dv), scale, causal)
    return fn


def test_dequantized_pins_reject_planted_mistakes(monkeypatch):
    assert _pins_pass(fp8.attention_dequantized, monkeypatch)
    for kind in ("axis", "dk_for_dq", "no_dv", "dv_for_dk"):
        assert not _pins_pass(_mutant(kind), monkeypatch), f"planted mistake {kind!r} passes every pin"
