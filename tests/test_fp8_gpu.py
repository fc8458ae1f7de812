"""FP8 forward with incoherent processing (fa_quantize_qk_fp8, fa_quantize_v_fp8,
fa_fwd_fp8) against the FP8 oracle (oracle/fp8.py):

* quantization is integer work, so the e4m3 codes and the per-head scales must match
  the oracle bit for bit (with and without the Hadamard rotation, d = 64 and 128);
* the forward pass on the codes is compared with the fp64 attention of the dequantized
  values.  L is computed from the fp32 scores and fp32 row sums and keeps the bf16
  tolerance.  O additionally carries the rounding of P to e4m3 (relative error at most
  2^-4 per element, unbiased): per row the error is a sum of independent
  +-2^-4 P_j v_j terms over l, so its RMS over the tensor is well below 2^-4 / sqrt(#
  keys that matter); the test bounds max |dO| <= 2^-3 and RMS(dO) <= 2^-6;
* incoherent processing must pay off: with outlier channels in Q and K, the rotated
  path's error against the exact attention of the original inputs must be several
  times smaller than the unrotated path's."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_tmem_gb300 import inputs
from gpu_helpers import TOL_L, to_dev
from oracle import fp8 as ofp8

pytestmark = pytest.mark.gpu

TOL_O8_MAX = 2.0 ** -3
TOL_O8_RMS = 2.0 ** -6


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    import exact_attention_tmem_gb300 as fa
    fa.build()
    torch.cuda.init()


def _signs(d, seed):
    rng = np.random.default_rng(seed)
    return rng.choice([-1.0, 1.0], size=d).astype(np.float32)


def _oracle_codes(x_bf16, signs):
    x = x_bf16.float().numpy()
    if signs is not None:
        x = ofp8.rotate(x, signs)
    vals, descale = ofp8.quantize(x)
    return ofp8.e4m3_code(vals), descale, vals


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("rotate", [False, True])
def test_qk_quantization_is_bit_exact(d, rotate):
    import exact_attention_tmem_gb300 as fa
    B, H, N = 2, 3, 300
    x = inputs.normal((B, H, N, d), 31000 + d)
    x = (x.float() * torch.linspace(0.5, 4.0, H).view(1, H, 1, 1)).to(torch.bfloat16)   # distinct head ranges
    x[0, 1, 7, 3] = 40.0                                                                   # an outlier
    s = _signs(d, 31001) if rotate else None
    x8, descale = fa.quantize_qk_fp8(x.cuda(), torch.from_numpy(s).cuda() if rotate else None)
    torch.cuda.synchronize()
    codes, ds_ref, _ = _oracle_codes(x, s)
    np.testing.assert_array_equal(descale.cpu().numpy(), ds_ref)
    got = x8.cpu().numpy()
    assert (got == codes).all(), f"{int((got != codes).sum())} of {codes.size} codes differ"


@pytest.mark.parametrize("N", [1, 17, 300])
def test_v_quantization_is_bit_exact_and_transposed(N):
    import exact_attention_tmem_gb300 as fa
    B, H, d = 1, 2, 128
    v = inputs.normal((B, H, N, d), 32000 + N)
    vt8, descale = fa.quantize_v_fp8(v.cuda())
    torch.cuda.synchronize()
    codes, ds_ref, _ = _oracle_codes(v, None)
    np.testing.assert_array_equal(descale.cpu().numpy(), ds_ref)
    got = vt8.cpu().numpy()
    npad = (N + 15) // 16 * 16
    assert got.shape == (B, H, d, npad)
    np.testing.assert_array_equal(got[..., :N], np.swapaxes(codes, -1, -2))
    assert (got[..., N:] == 0).all()


def _fp8_forward(q, k, v, causal, signs):
    import exact_attention_tmem_gb300 as fa
    sg = torch.from_numpy(signs).cuda() if signs is not None else None
    qd, kd, vd = to_dev(q, k, v)
    q8, dq = fa.quantize_qk_fp8(qd, sg)
    k8, dk = fa.quantize_qk_fp8(kd, sg)
    vt8, dv = fa.quantize_v_fp8(vd)
    o, lse = fa.fwd_fp8(q8, k8, vt8, dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _dequantized_reference(q, k, v, causal, signs, scale):
    _, dq, qv = _oracle_codes(q, signs)
    _, dk, kv = _oracle_codes(k, signs)
    _, dv, vv = _oracle_codes(v, None)
    return ofp8.attention_dequantized(qv, kv, vv, dq, dk, dv, scale, causal, oracle.attention_fwd)


CASES = [  # B, H, N
    (1, 1, 1), (1, 2, 17), (1, 2, 128), (2, 2, 129), (1, 3, 300), (2, 2, 513), (1, 2, 1000),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", CASES)
def test_fp8_forward_matches_dequantized_oracle(B, H, N, causal):
    d = 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = inputs.random_inputs(B, H, N, d, seed=33000 + B * 100 + H * 10 + N)
    s = _signs(d, 33001)
    o, lse = _fp8_forward(q, k, v, causal, s)
    O_ref, L_ref = _dequantized_reference(q, k, v, causal, s, scale)
    err = np.abs(o - O_ref)
    what = f"B={B} H={H} N={N} causal={causal}"
    assert err.max() <= TOL_O8_MAX, f"{what}: max |dO| {err.max():.3e}"
    assert math.sqrt((err ** 2).mean()) <= TOL_O8_RMS, f"{what}: rms dO {math.sqrt((err ** 2).mean()):.3e}"
    assert np.abs(lse - L_ref).max() <= TOL_L, f"{what}: max |dL| {np.abs(lse - L_ref).max():.3e}"


def test_fp8_forward_grouped_query():
    import exact_attention_tmem_gb300 as fa
    B, H, Hkv, N, d = 1, 4, 2, 400, 128
    q = inputs.normal((B, H, N, d), 34000)
    k = inputs.normal((B, Hkv, N, d), 34001)
    v = inputs.normal((B, Hkv, N, d), 34002)
    s = _signs(d, 34003)
    o, lse = _fp8_forward(q, k, v, True, s)
    k_rep, v_rep = k.repeat_interleave(2, dim=1), v.repeat_interleave(2, dim=1)
    O_ref, L_ref = _dequantized_reference(q, k_rep, v_rep, True, s, 1.0 / math.sqrt(d))
    assert np.abs(o - O_ref).max() <= TOL_O8_MAX
    assert np.abs(lse - L_ref).max() <= TOL_L


def test_incoherent_processing_reduces_the_error():
    """Outlier channels in Q and K: the Hadamard rotation must cut the error of the FP8
    result against the exact attention of the original (unquantized) inputs."""
    B, H, N, d = 1, 4, 512, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (inputs.normal((B, H, N, d), 35000 + i).float() for i in range(3))
    ch = torch.tensor([3, 50, 91])
    q[..., ch] *= 12.0
    k[..., ch] *= 12.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    f = inputs.as_f64
    O_exact, _ = oracle.attention_fwd(f(q), f(k), f(v), scale, False)
    o_rot, _ = _fp8_forward(q, k, v, False, _signs(d, 35003))
    o_plain, _ = _fp8_forward(q, k, v, False, None)
    rms = lambda a: math.sqrt(((a - O_exact) ** 2).mean())
    assert rms(o_rot) < 0.5 * rms(o_plain), f"rotated {rms(o_rot):.3e} vs plain {rms(o_plain):.3e}"
