"""fp64 oracle for decoding: one query row per head against a long key/value sequence.

TEST INFRASTRUCTURE ONLY, like the rest of this package: only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it; the CUDA
library never does, and the two share no code.

What it computes.  For each batch b and query head h, with key/value head
kv = h // (H / Hkv) (grouped-query attention; Hkv = H is plain multi-head attention):

    s_j = scale * q[b, h] . k[b, kv, j]          j = 0 .. Nk-1
    O[b, h] = sum_j softmax(s)_j v[b, kv, j],    L[b, h] = log sum_j exp(s_j)

The decode query is the newest position, so it sees every key and no mask applies.

Sources:
  * "FlashAttention" deep dive, section "Implementation notes": decoding with a single
    query row is parallelised over chunks of the keys; each chunk gives a partial
    (m, l, acc) triple and the triples are merged with the same rescaling rule the
    tiled forward pass uses.  ``decode_split`` follows those steps.
  * "Flash Attention and Memory-Efficient Attention Variants", section "Worked example:
    tracing the running statistics by hand": one query against four keys in two tiles
    of two keys, with the running max, denominator and unnormalised output printed
    after each tile (the pins in tests/test_oracle_decode.py).

Inputs are float64 arrays (already rounded to the values the GPU receives):
q [B, H, d], k and v [B, Hkv, Nk, d].  Results are float64.
"""
from __future__ import annotations

import numpy as np


def _kv_index(H: int, Hkv: int) -> np.ndarray:
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError("the query heads must be a multiple of the key/value heads")
    return np.arange(H) // (H // Hkv)


def attention_decode(q, k, v, scale: float):
    """The plain definition: softmax of the scaled scores, then the weighted sum of V.
    Returns (O [B, H, d], L [B, H]) with L the natural-log logsumexp of the scores."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, d = q.shape
    kv = _kv_index(H, k.shape[1])
    O = np.empty((B, H, d))
    L = np.empty((B, H))
    for b in range(B):
        for h in range(H):
            s = scale * (k[b, kv[h]] @ q[b, h])          # [Nk]
            m = s.max()
            e = np.exp(s - m)                            # max-subtracted: same value, no overflow
            l = e.sum()
            O[b, h] = (e @ v[b, kv[h]]) / l
            L[b, h] = m + np.log(l)
    return O, L


def chunk_partial(q, k, v, scale: float):
    """One chunk of keys for one head: the running statistics after that chunk alone,
    m = max_j s_j, l = sum_j exp(s_j - m), acc = sum_j exp(s_j - m) v_j (unnormalised)."""
    s = scale * (np.asarray(k, dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ np.asarray(v, dtype=np.float64)


def merge(partials):
    """Merge (m, l, acc) triples: rescale each to the common max m* by exp(m_c - m*)
    and add.  Returns the merged (m*, l*, acc*)."""
    m = max(p[0] for p in partials)
    l = sum(p[1] * np.exp(p[0] - m) for p in partials)
    acc = sum(p[2] * np.exp(p[0] - m) for p in partials)
    return m, l, acc


def decode_split(q, k, v, scale: float, chunk: int):
    """Split-key decoding in the pages' steps: partial triples per chunk of `chunk`
    keys, merged, then O = acc / l and L = m + log l."""
    if chunk < 1:
        raise ValueError("chunk must be positive")
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    B, H, d = q.shape
    Nk = k.shape[2]
    kv = _kv_index(H, k.shape[1])
    O = np.empty((B, H, d))
    L = np.empty((B, H))
    for b in range(B):
        for h in range(H):
            parts = [chunk_partial(q[b, h], k[b, kv[h], c:c + chunk], v[b, kv[h], c:c + chunk], scale)
                     for c in range(0, Nk, chunk)]
            m, l, acc = merge(parts)
            O[b, h] = acc / l
            L[b, h] = m + np.log(l)
    return O, L
