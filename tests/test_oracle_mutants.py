"""Each plausible mistake, planted in a copy of the oracle, must fail at least one pin.

The mutants are compiled from fa_oracle.c with one textual edit each, into a
temporary directory; the real oracle is untouched.  This shows that the pins
are strong enough to catch a dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the oracle.
"""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "fa_oracle.c")

MUTANTS = {
    "scores without scale": ("s *= scale;", ";"),
    "causal mask off by one": ("return causal ? (i + 1 < n ? i + 1 : n) : n;",
                               "return causal ? (i < n ? i : n) : n;"),
    "causal mask one too wide": ("return causal ? (i + 1 < n ? i + 1 : n) : n;",
                                 "return causal ? (i + 2 < n ? i + 2 : n) : n;"),
    "logsumexp without max": ("*lse_out = mx + log(z);", "*lse_out = log(z);"),
    "softmax not normalised": ("for (long j = 0; j < nk; ++j) p[j] /= z;", ";"),
    "values reversed": ("const double *vj = vh + j * d;\n        double pj",
                        "const double *vj = vh + (nk - 1 - j) * d;\n        double pj"),
    "D term dropped": ("dp[j] = p[j] * (s - di);", "dp[j] = p[j] * s;"),
    "dS sign flipped": ("dp[j] = p[j] * (s - di);", "dp[j] = p[j] * (di - s);"),
    "dP uses Q instead of V": ("for (long t = 0; t < d; ++t) s += doi[t] * vj[t];",
                               "for (long t = 0; t < d; ++t) s += doi[t] * qi[t];"),
    "dQ without scale": ("for (long t = 0; t < d; ++t) dqi[t] *= scale;", ";"),
    "dQ uses V instead of K": ("const double *kj = kh + j * d;\n                    for (long t = 0; t < d; ++t) dqi[t]",
                               "const double *kj = vh + j * d;\n                    for (long t = 0; t < d; ++t) dqi[t]"),
    "dK without scale": ("double a = scale * dp[j], b = p[j];", "double a = dp[j], b = p[j];"),
    "dK uses dO instead of Q": ("dkj[t] += a * qi[t];", "dkj[t] += a * doi[t];"),
    "dV uses Q instead of dO": ("dvj[t] += b * doi[t];", "dvj[t] += b * qi[t];"),
    "dV transposed (P_ji)": ("double a = scale * dp[j], b = p[j];",
                             "double a = scale * dp[j], b = (j < nk ? p[nk - 1 - j] : 0.0);"),
    "D from V instead of O": ("for (long t = 0; t < d; ++t) di += doi[t] * oi[t];",
                              "for (long t = 0; t < d; ++t) di += doi[t] * vh[i * d + t];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not unique in fa_oracle.c"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutant_src), out=str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, RuntimeError, FloatingPointError) as e:
            caught.append(f"{pin.__name__}: {str(e)[:80]}")
    assert caught, f"planted mistake '{name}' passed every pin"
