"""Pins for the decoding oracle (oracle/decode.py), checked against what the pages and the
mathematics fix: the worked example's printed numbers (one query, four keys, two tiles),
an independent implementation (the C oracle's last causal row), closed forms, the
grouped-query mapping and invariance under the chunking.  No GPU."""
import math

import numpy as np
import pytest

import oracle
from oracle import decode

GOLDEN = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rhs = (x.strip() for x in line.split("="))
        vals[key] = np.array([float(t) for t in rhs.split()])
    q = vals["q"][None, None, :]
    K = np.stack([vals[f"K{i}"] for i in range(4)])[None, None]
    V = np.stack([vals[f"V{i}"] for i in range(4)])[None, None]
    return q, K, V, vals


def test_worked_example_output():
    q, K, V, g = _golden()
    O, L = decode.attention_decode(q, K, V, float(g["scale"][0]))
    np.testing.assert_allclose(O[0, 0], g["O"], atol=5e-9)
    # L = log(e^1 + e^0 + e^3 + e^-1)
    assert abs(L[0, 0] - math.log(math.e + 1 + math.e ** 3 + math.e ** -1)) < 1e-12


def test_worked_example_tile_states():
    """Keys {0, 1} and {2, 3} as two chunks: the first chunk's triple and the merged
    denominator are the values the page prints after tile 1 and tile 2."""
    q, K, V, g = _golden()
    p1 = decode.chunk_partial(q[0, 0], K[0, 0, :2], V[0, 0, :2], 1.0)
    assert p1[0] == g["m_tile1"][0]
    assert abs(p1[1] - g["l_tile1"][0]) < 5e-5
    np.testing.assert_allclose(p1[2], g["Oacc_tile1"], atol=5e-5)
    p2 = decode.chunk_partial(q[0, 0], K[0, 0, 2:], V[0, 0, 2:], 1.0)
    m, l, acc = decode.merge([p1, p2])
    assert m == g["m_final"][0]
    assert abs(math.exp(p1[0] - m) - g["c_tile2"][0]) < 5e-6
    assert abs(l - g["l_final"][0]) < 5e-6
    # the page computes this line from its rounded tile-1 numbers (0.13534 x 3.4715 ...),
    # so its last printed digit can be one off
    np.testing.assert_allclose(acc, g["Oacc_tile2"], atol=1.5e-4)
    O, _ = decode.decode_split(q, K, V, 1.0, chunk=2)
    np.testing.assert_allclose(O[0, 0], g["O"], atol=5e-9)


@pytest.mark.parametrize("Nk,d", [(1, 4), (7, 16), (300, 64)])
def test_matches_last_causal_row_of_the_c_oracle(Nk, d):
    """An independent implementation: the C oracle's causal forward, restricted to its
    last row, is the decode of that row's query against every key."""
    rng = np.random.default_rng(Nk + d)
    B, H = 2, 3
    Q = rng.standard_normal((B, H, Nk, d))
    K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d))
    scale = 1.0 / math.sqrt(d)
    O_ref, L_ref = oracle.attention_fwd_rows(Q, K, V, scale, True, np.array([Nk - 1]))
    O, L = decode.attention_decode(Q[:, :, -1], K, V, scale)
    np.testing.assert_allclose(O, O_ref[:, :, 0], atol=1e-12)
    np.testing.assert_allclose(L, L_ref[:, :, 0], atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(5)
    d = 8
    q = rng.standard_normal((1, 1, d))
    kvec = rng.standard_normal(d)
    V = rng.standard_normal((1, 1, 10, d))
    K = np.broadcast_to(kvec, (1, 1, 10, d)).copy()       # identical keys: uniform weights
    O, L = decode.attention_decode(q, K, V, 0.3)
    np.testing.assert_allclose(O[0, 0], V[0, 0].mean(axis=0), atol=1e-12)
    assert abs(L[0, 0] - (0.3 * q[0, 0] @ kvec + math.log(10))) < 1e-12
    O1, L1 = decode.attention_decode(q, K[:, :, :1], V[:, :, :1], 0.3)   # one key
    np.testing.assert_allclose(O1[0, 0], V[0, 0, 0], atol=1e-15)
    assert abs(L1[0, 0] - 0.3 * q[0, 0] @ kvec) < 1e-12


def test_grouped_query_mapping():
    rng = np.random.default_rng(9)
    B, H, Hkv, Nk, d = 2, 6, 2, 33, 16
    q = rng.standard_normal((B, H, d))
    K = rng.standard_normal((B, Hkv, Nk, d))
    V = rng.standard_normal((B, Hkv, Nk, d))
    O, L = decode.attention_decode(q, K, V, 0.25)
    O_rep, L_rep = decode.attention_decode(q, np.repeat(K, 3, axis=1), np.repeat(V, 3, axis=1), 0.25)
    np.testing.assert_array_equal(O, O_rep)
    np.testing.assert_array_equal(L, L_rep)
    # query head 4 uses key/value head 1
    o4, l4 = decode.attention_decode(q[:, 4:5], K[:, 1:2], V[:, 1:2], 0.25)
    np.testing.assert_array_equal(O[:, 4], o4[:, 0])


@pytest.mark.parametrize("chunk", [1, 3, 64, 1000])
def test_chunking_does_not_change_the_result(chunk):
    rng = np.random.default_rng(chunk)
    B, H, Nk, d = 1, 2, 257, 32
    q = 3.0 * rng.standard_normal((B, H, d))              # peaked rows exercise the rescale
    K = rng.standard_normal((B, H, Nk, d))
    V = rng.standard_normal((B, H, Nk, d))
    O, L = decode.attention_decode(q, K, V, 0.5)
    Os, Ls = decode.decode_split(q, K, V, 0.5, chunk)
    np.testing.assert_allclose(Os, O, atol=1e-12)
    np.testing.assert_allclose(Ls, L, atol=1e-12)


def test_merge_without_rescale_is_caught():
    """A merge that forgets the exp(m_c - m*) factor fails the tile-state pin."""
    q, K, V, g = _golden()
    p1 = decode.chunk_partial(q[0, 0], K[0, 0, :2], V[0, 0, :2], 1.0)
    p2 = decode.chunk_partial(q[0, 0], K[0, 0, 2:], V[0, 0, 2:], 1.0)
    wrong_l = p1[1] + p2[1]
    assert abs(wrong_l - g["l_final"][0]) > 1e-2
