"""Brute-force attention in 50-digit arithmetic (mpmath), for tiny inputs.

Used only to pin the fp64 oracle.  It shares nothing with the oracle: the
softmax is evaluated without the max subtraction, straight from the
definition exp(s_ij) / sum_j exp(s_ij), and the gradients come from central
finite differences of f = sum(O * dO) at 50 digits, not from the analytic
backward formulas.
"""
from __future__ import annotations

import mpmath as mp

mp.mp.dps = 50


def _to_mp(a):
    return [[x if isinstance(x, mp.mpf) else mp.mpf(float(x)) for x in row] for row in a]


def forward(q, k, v, scale, causal):
    """q, k, v: [N][d] nested lists (floats).  Returns (O, L) as mp numbers."""
    Q, K, V = _to_mp(q), _to_mp(k), _to_mp(v)
    n, d = len(Q), len(Q[0])
    sc = mp.mpf(scale)
    O, L = [], []
    for i in range(n):
        keys = range(i + 1) if causal else range(n)
        w = {j: mp.exp(sc * mp.fsum(Q[i][t] * K[j][t] for t in range(d))) for j in keys}
        z = mp.fsum(w.values())
        O.append([mp.fsum(w[j] * V[j][t] for j in keys) / z for t in range(d)])
        L.append(mp.log(z))
    return O, L


def objective(q, k, v, do, scale, causal):
    O, _ = forward(q, k, v, scale, causal)
    return mp.fsum(O[i][t] * mp.mpf(float(do[i][t])) for i in range(len(O)) for t in range(len(O[0])))


def gradients(q, k, v, do, scale, causal, h="1e-20"):
    """Central differences of sum(O*dO) w.r.t. every element of q, k, v."""
    h = mp.mpf(h)
    base = {"q": [list(map(mp.mpf, map(float, r))) for r in q],
            "k": [list(map(mp.mpf, map(float, r))) for r in k],
            "v": [list(map(mp.mpf, map(float, r))) for r in v]}
    grads = {}
    for name in ("q", "k", "v"):
        g = []
        for i in range(len(base[name])):
            row = []
            for t in range(len(base[name][0])):
                plus = {n: [r[:] for r in m] for n, m in base.items()}
                minus = {n: [r[:] for r in m] for n, m in base.items()}
                plus[name][i][t] += h
                minus[name][i][t] -= h
                fp = objective(plus["q"], plus["k"], plus["v"], do, scale, causal)
                fm = objective(minus["q"], minus["k"], minus["v"], do, scale, causal)
                row.append((fp - fm) / (2 * h))
            g.append(row)
        grads[name] = g
    return grads["q"], grads["k"], grads["v"]
