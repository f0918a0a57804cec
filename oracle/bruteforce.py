"""Pure-Python scalar brute force of the tensor-parallel FFN (tiny shapes only).

TEST INFRASTRUCTURE ONLY.  A second, independent writing of the oracle's
forms in plain Python loops (math.tanh / math.exp), used to cross-check the
C oracle on shapes of a few thousand multiply-adds.  It follows the same
passages: "7.9 Tensor and pipeline parallelism (TP, PP)", §2.1 "The FFN,
sharded" (column-shard W1, row-shard W2, sum the partials) and the SwiGLU
form of "S17 Tensor & Pipeline Parallelism", listing "the megatron pattern".
Shapes: x [N][d] (NONE: [N][d_ff]), W1/W3 [d_ff][d], W2 [d][d_ff].
"""
from __future__ import annotations

import math


def _gelu(u):
    return 0.5 * u * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (u + 0.044715 * u ** 3)))


def _silu(u):
    return u / (1.0 + math.exp(-u))


def ffn_sharded_forward(x, W1, W3, b1, W2, b2, T_p, act):
    """Returns (y, partials) as nested lists; partials[t][n][c]."""
    N = len(x)
    d = len(W2)
    d_ff = len(W2[0])
    s = d_ff // T_p
    partials = [[[0.0] * d for _ in range(N)] for _ in range(T_p)]
    y = [[0.0] * d for _ in range(N)]
    for n in range(N):
        for t in range(T_p):
            h = []
            for jj in range(s):
                j = t * s + jj
                if act == "none":
                    h.append(x[n][j])
                    continue
                z = 0.0
                for k in range(d):
                    z += W1[j][k] * x[n][k]
                if act == "swiglu":
                    g = 0.0
                    for k in range(d):
                        g += W3[j][k] * x[n][k]
                    h.append(_silu(z) * g)
                else:
                    if b1 is not None:
                        z += b1[j]
                    h.append(_gelu(z) if act == "gelu_tanh" else z)
            for c in range(d):
                acc = 0.0
                for jj in range(s):
                    acc += W2[c][t * s + jj] * h[jj]
                partials[t][n][c] = acc
        for c in range(d):
            acc = 0.0
            for t in range(T_p):
                acc += partials[t][n][c]
            if b2 is not None:
                acc += b2[c]
            y[n][c] = acc
    return y, partials
