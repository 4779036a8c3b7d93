"""Pure-Python loop versions of the oracle's kernels, for tiny inputs only.

These restate each definition element by element with the standard library's math (no NumPy
vectorisation, no library matmul), so that the vectorised oracle in `model.py` can be checked
against an independent formulation:
* attention: softmax(q k^T / sqrt D) v written as explicit sums;
* RoPE: each pair (x0, x1) as the complex number x0 + i x1 multiplied by e^{i theta};
* LayerNorm: the two-pass mean / variance as explicit sums.
"""
from __future__ import annotations

import cmath
import math


def attention_loops(q, k, v):
    """q, k, v: nested lists [L][nh][D] -> [L][nh][D]."""
    L, nh, D = len(q), len(q[0]), len(q[0][0])
    out = [[[0.0] * D for _ in range(nh)] for _ in range(L)]
    for h in range(nh):
        for i in range(L):
            sc = []
            for j in range(L):
                acc = 0.0
                for d in range(D):
                    acc += q[i][h][d] * k[j][h][d]
                sc.append(acc / math.sqrt(D))
            m = max(sc)
            e = [math.exp(s - m) for s in sc]
            z = sum(e)
            for d in range(D):
                out[i][h][d] = sum(e[j] * v[j][h][d] for j in range(L)) / z
    return out


def rope_loops(x, pos, base=10000.0):
    """x: [L][nh][D] nested lists, pos: [L][3].  Axis blocks (D/8, 7D/16, 7D/16)."""
    L, nh, D = len(x), len(x[0]), len(x[0][0])
    widths = (D // 8, 7 * D // 16, 7 * D // 16)
    out = [[list(row) for row in tok] for tok in x]
    for i in range(L):
        for h in range(nh):
            off = 0
            for a, d in enumerate(widths):
                for j in range(d // 2):
                    theta = pos[i][a] * base ** (-2.0 * j / d)
                    zc = complex(x[i][h][off + 2 * j], x[i][h][off + 2 * j + 1])
                    zr = zc * cmath.exp(1j * theta)
                    out[i][h][off + 2 * j] = zr.real
                    out[i][h][off + 2 * j + 1] = zr.imag
                off += d
    return out


def layer_norm_loops(row, eps=1e-6):
    n = len(row)
    mu = sum(row) / n
    var = sum((a - mu) ** 2 for a in row) / n
    return [(a - mu) / math.sqrt(var + eps) for a in row]
