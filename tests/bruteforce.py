"""A second, independently written attention reference for tiny inputs.

Pure Python loops over nested lists: RoPE as multiplication of the complex
number x_{2i} + i*x_{2i+1} by e^{i*pos*theta_i}, scores as explicit sums, the
mask as explicit position tests, softmax with math.exp.  It shares nothing with
oracle/attention.py (no numpy, no matrix helper), so an error in either shows
up as a disagreement between the two.
"""
from __future__ import annotations

import cmath
import math


def rotate_complex(vec, pos, base, offset=0, dims=None):
    """Rotate pairs (offset+2i, offset+2i+1) of vec by pos*base^(-2i/dims)."""
    vec = list(vec)
    dims = len(vec) - offset if dims is None else dims
    for i in range(dims // 2):
        theta = math.exp(-2.0 * i / dims * math.log(base))
        z = complex(vec[offset + 2 * i], vec[offset + 2 * i + 1]) * cmath.exp(1j * pos * theta)
        vec[offset + 2 * i], vec[offset + 2 * i + 1] = z.real, z.imag
    return vec


def visible(pos_q, n, causal, window, n_sink):
    if causal and n > pos_q:
        return False
    if window > 0 and pos_q - n >= window and n >= n_sink:
        return False
    return True


def attend_one(qvec, keys, values, pos_q, scale, causal=True, window=0, n_sink=0):
    """Output and natural-log normaliser for one query over lists of keys/values."""
    scores = []
    for n, kvec in enumerate(keys):
        if visible(pos_q, n, causal, window, n_sink):
            acc = 0.0
            for a, b in zip(qvec, kvec):
                acc += a * b
            scores.append((n, acc * scale))
    top = max(s for _, s in scores)
    weights = [(n, math.exp(s - top)) for n, s in scores]
    total = sum(w for _, w in weights)
    out = [0.0] * len(values[0])
    for n, w in weights:
        for d in range(len(out)):
            out[d] += (w / total) * values[n][d]
    return out, top + math.log(total)


def prefill(q, k, v, rope_base, scale, causal=True, q_offset=0, window=0, n_sink=0):
    """q [S_q][n_h][D], k/v [S_k][n_kv][D] nested lists (one batch entry).
    Returns out [S_q][n_h][D_v] and lse [n_h][S_q]."""
    S_q, n_h = len(q), len(q[0])
    S_k, n_kv = len(k), len(k[0])
    out = [[None] * n_h for _ in range(S_q)]
    lse = [[None] * S_q for _ in range(n_h)]
    for h in range(n_h):
        g = (h * n_kv) // n_h
        keys = []
        for n in range(S_k):
            kv = k[n][g]
            keys.append(rotate_complex(kv, n, rope_base) if rope_base > 0 else list(kv))
        values = [list(v[n][g]) for n in range(S_k)]
        for m in range(S_q):
            pos = q_offset + m
            qv = rotate_complex(q[m][h], pos, rope_base) if rope_base > 0 else list(q[m][h])
            out[m][h], lse[h][m] = attend_one(qv, keys, values, pos, scale, causal, window, n_sink)
    return out, lse
