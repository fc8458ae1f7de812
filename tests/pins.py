"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when
the oracle disagrees with the pages or with mathematics.  They are run on the
real oracle (tests/test_oracle_pins.py) and on copies of it with a planted
mistake (tests/test_oracle_mutants.py), where at least one must fail.
"""
from __future__ import annotations

import math
import os

import numpy as np

import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rhs = line.split("=", 1)
            vals[key.strip()] = np.array([float(x) for x in rhs.split()])
    return vals


def _h(x):
    """[N, d] -> [1, 1, N, d]"""
    return np.asarray(x, dtype=np.float64)[None, None]


def _close(a, b, atol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert np.all(np.isfinite(a)) and err <= atol, f"{what}: max|diff| = {err:.3e} > {atol:.1e}"


# --- the worked example ("Flash Attention and Memory-Efficient Attention Variants",
#     section "Worked example: tracing the running statistics by hand") -------------

def _example():
    g = read_golden("worked_example.txt")
    K = np.stack([g["K0"], g["K1"], g["K2"], g["K3"]])
    V = np.stack([g["V0"], g["V1"], g["V2"], g["V3"]])
    return g, K, V


def pin_worked_example_output(orc):
    """Final output and full-row denominator printed by the page (scale 1)."""
    g, K, V = _example()
    Q = np.zeros((4, 2))
    Q[0] = g["q"]
    o, lse = orc.attention_fwd(_h(Q), _h(K), _h(V), float(g["scale"][0]), False)
    _close(o[0, 0, 0], g["O"], 5e-9, "worked example O")
    # page: l = 1.20344 relative to the final running max m = 3, so L = m + ln(l)
    _close(lse[0, 0, 0], g["m_final"][0] + math.log(g["l_final"][0]), 5e-6, "worked example L")


def pin_worked_example_probabilities(orc):
    """The page's softmax row [0.1125, 0.0414, 0.8310, 0.0152], read out with V = I."""
    g, K, V = _example()
    Q4 = np.zeros((4, 4))
    Q4[0, :2] = g["q"]
    K4 = np.zeros((4, 4))
    K4[:, :2] = K
    o, _ = orc.attention_fwd(_h(Q4), _h(K4), _h(np.eye(4)), 1.0, False)
    _close(o[0, 0, 0], g["P"], 5e-5, "worked example softmax row")


def pin_worked_example_tile_states(orc):
    """State after tile 1 (keys 0-1) and the tile-2 update, as printed on the page."""
    g, K, V = _example()
    Q = np.array([g["q"], g["q"]])
    o, lse = orc.attention_fwd(_h(Q), _h(K[:2]), _h(V[:2]), 1.0, False)
    # after tile 1: running max 1, l = 1.3679, unnormalised O = [2.1036, 3.4715]
    l1 = math.exp(lse[0, 0, 0] - g["m_tile1"][0])
    _close(l1, g["l_tile1"][0], 5e-5, "tile-1 denominator")
    _close(o[0, 0, 0] * l1, g["Oacc_tile1"], 5e-5, "tile-1 unnormalised output")
    # tile 2: correction exp(1 - 3) rescales tile 1's accumulator; adding tile 2 gives
    # the unnormalised [5.4129, 6.6164] relative to m = 3
    c = math.exp(g["m_tile1"][0] - g["m_final"][0])
    _close(c, g["c_tile2"][0], 5e-6, "tile-2 correction factor")
    Q1 = np.zeros((4, 2))
    Q1[0] = g["q"]
    o_all, lse_all = orc.attention_fwd(_h(Q1), _h(K), _h(V), 1.0, False)
    l2 = math.exp(lse_all[0, 0, 0] - g["m_final"][0])
    _close(o_all[0, 0, 0] * l2, g["Oacc_tile2"], 5e-4, "tile-2 unnormalised output")


# --- brute force at 50 digits --------------------------------------------------------

def _tiny_cases():
    rng = np.random.default_rng(7)
    cases = []
    for n, d, causal, scale in [(1, 2, False, 0.7), (3, 2, True, 1.0), (4, 3, False, 0.5),
                                (5, 3, True, 0.9), (6, 2, False, 1.3), (7, 2, True, 0.35)]:
        q, k, v, do = (rng.standard_normal((n, d)) * 1.5 for _ in range(4))
        cases.append((q, k, v, do, scale, causal))
    return cases


def pin_brute_force_forward(orc):
    """O and L against 50-digit evaluation of exp(s)/sum exp(s) (no max subtraction)."""
    for q, k, v, _, scale, causal in _tiny_cases():
        o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), scale, causal)
        O, L = brute.forward(q, k, v, scale, causal)
        _close(o[0, 0], np.array(O, dtype=np.float64), 1e-13, f"brute O (n={len(q)}, causal={causal})")
        _close(lse[0, 0], np.array(L, dtype=np.float64), 1e-13, f"brute L (n={len(q)}, causal={causal})")


def pin_brute_force_gradients(orc):
    """dQ, dK, dV against 50-digit central differences of sum(O * dO)."""
    for q, k, v, do, scale, causal in _tiny_cases()[:4]:
        dq, dk, dv = orc.attention_bwd(_h(q), _h(k), _h(v), _h(do), scale, causal)
        gq, gk, gv = brute.gradients(q, k, v, do, scale, causal)
        for name, a, b in (("dQ", dq, gq), ("dK", dk, gk), ("dV", dv, gv)):
            _close(a[0, 0], np.array(b, dtype=np.float64), 1e-11,
                   f"brute {name} (n={len(q)}, causal={causal})")


# --- closed forms and invariants -------------------------------------------------------

def pin_zero_queries(orc):
    """Q = 0: every visible key gets equal weight.  L = ln N (full), ln(i+1) (causal),
    and causal O_i is the mean of V_0..V_i."""
    rng = np.random.default_rng(11)
    n, d = 9, 4
    q = np.zeros((n, d))
    k, v = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), 0.5, False)
    _close(lse[0, 0], np.full(n, math.log(n)), 1e-14, "L = ln N for Q = 0")
    _close(o[0, 0], np.tile(v.mean(axis=0), (n, 1)), 1e-14, "O = mean V for Q = 0")
    o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), 0.5, True)
    _close(lse[0, 0], np.log(np.arange(1, n + 1)), 1e-14, "causal L_i = ln(i+1)")
    want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    _close(o[0, 0], want, 1e-14, "causal O_i = mean V_0..V_i")


def pin_constant_values(orc):
    """All V rows equal v: O = v for every row, whatever the scores."""
    rng = np.random.default_rng(12)
    n, d = 8, 5
    q, k = rng.standard_normal((n, d)) * 3, rng.standard_normal((n, d)) * 3
    vrow = rng.standard_normal(d)
    v = np.tile(vrow, (n, 1))
    for causal in (False, True):
        o, _ = orc.attention_fwd(_h(q), _h(k), _h(v), 0.8, causal)
        _close(o[0, 0], v, 1e-14, f"O = v (causal={causal})")


def pin_single_key(orc):
    """N = 1: O = V_0 and L = scale * q.k; causal row 0 likewise sees only key 0."""
    rng = np.random.default_rng(13)
    q, k, v = (rng.standard_normal((1, 6)) for _ in range(3))
    o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), 0.3, False)
    _close(o[0, 0, 0], v[0], 1e-15, "N=1 output")
    _close(lse[0, 0, 0], 0.3 * float(q[0] @ k[0]), 1e-14, "N=1 logsumexp")
    q, k, v = (rng.standard_normal((5, 6)) for _ in range(3))
    o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), 0.3, True)
    _close(o[0, 0, 0], v[0], 1e-15, "causal row 0 output")
    _close(lse[0, 0, 0], 0.3 * float(q[0] @ k[0]), 1e-14, "causal row 0 logsumexp")


def pin_rows_sum_to_one(orc):
    """A column of ones in V reads back sum_j P_ij, which must be 1."""
    rng = np.random.default_rng(14)
    n, d = 10, 3
    q, k, v = rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d)) * 2, rng.standard_normal((n, d))
    v[:, 1] = 1.0
    for causal in (False, True):
        o, _ = orc.attention_fwd(_h(q), _h(k), _h(v), 1.1, causal)
        _close(o[0, 0, :, 1], np.ones(n), 1e-14, f"row sums of P (causal={causal})")


def pin_key_shift(orc):
    """Adding one vector c to every key row shifts row i's scores by scale*q_i.c:
    O is unchanged and L_i grows by exactly that amount."""
    rng = np.random.default_rng(15)
    n, d, scale = 7, 4, 0.6
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    c = rng.standard_normal(d)
    for causal in (False, True):
        o1, l1 = orc.attention_fwd(_h(q), _h(k), _h(v), scale, causal)
        o2, l2 = orc.attention_fwd(_h(q), _h(k + c), _h(v), scale, causal)
        _close(o2, o1, 1e-13, f"O under key shift (causal={causal})")
        _close(l2[0, 0] - l1[0, 0], scale * (q @ c), 1e-13, f"L under key shift (causal={causal})")


def pin_gradient_sums(orc):
    """sum_j dV_j = sum_i dO_i (rows of P sum to 1) and sum_j dK_j = 0
    (sum_j dS_ij = O_i.dO_i - D_i = 0)."""
    rng = np.random.default_rng(16)
    n, d = 9, 4
    q, k, v, do = (rng.standard_normal((n, d)) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(_h(q), _h(k), _h(v), _h(do), 0.7, causal)
        _close(dv[0, 0].sum(axis=0), do.sum(axis=0), 1e-13, f"sum dV (causal={causal})")
        _close(dk[0, 0].sum(axis=0), np.zeros(d), 1e-13, f"sum dK (causal={causal})")


def pin_finite_differences(orc):
    """Analytic dQ, dK, dV against fp64 central differences (h = 1e-6) of
    f = sum(O * dO), for N up to 16."""
    rng = np.random.default_rng(17)
    for n, d, causal in [(5, 3, False), (16, 4, True), (12, 3, False)]:
        q, k, v, do = (rng.standard_normal((1, 2, n, d)) for _ in range(4))
        scale = 0.45
        dq, dk, dv = orc.attention_bwd(q, k, v, do, scale, causal)

        def f(qq, kk, vv):
            o, _ = orc.attention_fwd(qq, kk, vv, scale, causal)
            return float(np.sum(o * do))

        h = 1e-6
        for name, x, g in (("dQ", q, dq), ("dK", k, dk), ("dV", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [xp if name == "dQ" else q, xp if name == "dK" else k, xp if name == "dV" else v]
                args_m = [xm if name == "dQ" else q, xm if name == "dK" else k, xm if name == "dV" else v]
                num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
            tol = 1e-7 * max(1.0, float(np.max(np.abs(num))))
            _close(g, num, tol, f"finite differences {name} (n={n}, causal={causal})")


# --- the page's tiled algorithm as an independent formulation --------------------------

def page_generator(n, d, seed):
    """Deterministic inputs of the deep-dive page's test: ((i*7919 + seed) % 1000)/500 - 1."""
    i = np.arange(n * d, dtype=np.int64)
    return (((i * 7919 + seed) % 1000).astype(np.float64) / 500.0 - 1.0).reshape(n, d)


def tiled_online_softmax(q, k, v, scale, bm, bn):
    """The deep-dive page's loop ("FlashAttention", section "How it works"), in fp64:
    running max m, running sum l, unnormalised accumulator, one divide at the end."""
    n, d = q.shape
    out, lse = np.zeros((n, d)), np.zeros(n)
    for i0 in range(0, n, bm):
        qi = q[i0:i0 + bm]
        m = np.full(qi.shape[0], -np.inf)
        l = np.zeros(qi.shape[0])
        acc = np.zeros((qi.shape[0], d))
        for j0 in range(0, n, bn):
            s = (qi @ k[j0:j0 + bn].T) * scale
            m_new = np.maximum(m, s.max(axis=1))
            p = np.exp(s - m_new[:, None])
            alpha = np.exp(m - m_new)
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[j0:j0 + bn]
            m = m_new
        out[i0:i0 + bm] = acc / l[:, None]
        lse[i0:i0 + bm] = m + np.log(l)
    return out, lse


def pin_page_tiled_case(orc):
    """n = 300 (not a multiple of the 64x64 tiles), d = 64, the page's input recipe:
    the oracle must agree with the tiled online-softmax loop."""
    n, d = 300, 64
    q, k, v = page_generator(n, d, 1), page_generator(n, d, 2), page_generator(n, d, 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.attention_fwd(_h(q), _h(k), _h(v), scale, False)
    t_o, t_l = tiled_online_softmax(q, k, v, scale, 64, 64)
    _close(o[0, 0], t_o, 1e-12, "tiled vs oracle O (n=300)")
    _close(lse[0, 0], t_l, 1e-12, "tiled vs oracle L (n=300)")


def pin_sampled_rows_match_full(orc):
    """The sampled-row entry point returns exactly the full forward's rows."""
    rng = np.random.default_rng(18)
    q, k, v = (rng.standard_normal((2, 3, 33, 8)) for _ in range(3))
    rows = np.array([0, 5, 17, 32])
    for causal in (False, True):
        o, l = orc.attention_fwd(q, k, v, 0.3, causal)
        o_r, l_r = orc.attention_fwd_rows(q, k, v, 0.3, causal, rows)
        _close(o_r, o[:, :, rows], 0.0, f"sampled rows O (causal={causal})")
        _close(l_r, l[:, :, rows], 0.0, f"sampled rows L (causal={causal})")


def pin_sampled_backward_rows(orc):
    """The row-sampled backward: all rows listed gives the full gradients, and the
    dK/dV contributions of disjoint row sets add up."""
    rng = np.random.default_rng(19)
    q, k, v, do = (rng.standard_normal((1, 2, 21, 5)) for _ in range(4))
    all_rows = np.arange(21)
    a, b = np.array([0, 3, 7, 20]), np.array([1, 2, 4, 5, 6] + list(range(8, 20)))
    for causal in (False, True):
        dq, dk, dv = orc.attention_bwd(q, k, v, do, 0.4, causal)
        dq_r, dk_r, dv_r = orc.attention_bwd_rows(q, k, v, do, 0.4, causal, all_rows)
        _close(dq_r, dq, 0.0, "row-sampled dQ, all rows")
        _close(dk_r, dk, 0.0, "row-sampled dK, all rows")
        _close(dv_r, dv, 0.0, "row-sampled dV, all rows")
        dq_a, dk_a, dv_a = orc.attention_bwd_rows(q, k, v, do, 0.4, causal, a)
        dq_b, dk_b, dv_b = orc.attention_bwd_rows(q, k, v, do, 0.4, causal, b)
        _close(dq_a, dq[:, :, a], 0.0, "row-sampled dQ rows")
        _close(dk_a + dk_b, dk, 1e-13, "dK contributions add up")
        _close(dv_a + dv_b, dv, 1e-13, "dV contributions add up")


ALL_PINS = [
    pin_worked_example_output,
    pin_worked_example_probabilities,
    pin_worked_example_tile_states,
    pin_brute_force_forward,
    pin_brute_force_gradients,
    pin_zero_queries,
    pin_constant_values,
    pin_single_key,
    pin_rows_sum_to_one,
    pin_key_shift,
    pin_gradient_sums,
    pin_finite_differences,
    pin_page_tiled_case,
    pin_sampled_rows_match_full,
    pin_sampled_backward_rows,
]
