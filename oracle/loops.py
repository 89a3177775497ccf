"""Brute-force scalar attention in pure Python loops (tiny inputs only).

TEST INFRASTRUCTURE ONLY. A second, independent spelling of the same
definition as ``attention.py`` (standard attention and its analytic gradient,
FlashAttention milestone page (nlp-lineage), "The notation"), written with
scalar loops and ``math.exp`` so that it shares no vectorised expression with
the NumPy oracle. It serves as a pin for the NumPy oracle on N <= 16.
"""
from __future__ import annotations

import math


def _allowed(i, j, causal, kv_len_b, block_mask, tile):
    if causal and j > i:
        return False
    if kv_len_b is not None and j >= kv_len_b:
        return False
    if block_mask is not None and not block_mask[i // tile][j // tile]:
        return False
    return True


def loop_attention_fwd_bwd(q, k, v, do, scale, causal=False, kv_len_b=None,
                           block_mask=None, tile=128):
    """One head. q, k, v, do: lists of N rows of d floats.

    Returns dict(O, LSE, dQ, dK, dV) as nested lists.
    """
    N = len(q)
    d = len(q[0])
    O = [[0.0] * d for _ in range(N)]
    LSE = [0.0] * N
    P = [[0.0] * N for _ in range(N)]
    for i in range(N):
        scores = []
        for j in range(N):
            if _allowed(i, j, causal, kv_len_b, block_mask, tile):
                s = 0.0
                for c in range(d):
                    s += q[i][c] * k[j][c]
                scores.append((j, scale * s))
        if not scores:
            LSE[i] = -math.inf
            continue
        mx = max(s for _, s in scores)
        tot = 0.0
        for _, s in scores:
            tot += math.exp(s - mx)
        LSE[i] = mx + math.log(tot)
        for j, s in scores:
            P[i][j] = math.exp(s - LSE[i])
        for c in range(d):
            acc = 0.0
            for j in range(N):
                acc += P[i][j] * v[j][c]
            O[i][c] = acc
    # backward of L = sum_ic dO_ic O_ic
    dV = [[0.0] * d for _ in range(N)]
    for j in range(N):
        for c in range(d):
            acc = 0.0
            for i in range(N):
                acc += P[i][j] * do[i][c]
            dV[j][c] = acc
    dS = [[0.0] * N for _ in range(N)]
    for i in range(N):
        Di = 0.0
        for c in range(d):
            Di += do[i][c] * O[i][c]
        for j in range(N):
            dp = 0.0
            for c in range(d):
                dp += do[i][c] * v[j][c]
            dS[i][j] = P[i][j] * (dp - Di)
    dQ = [[0.0] * d for _ in range(N)]
    dK = [[0.0] * d for _ in range(N)]
    for i in range(N):
        for c in range(d):
            acc = 0.0
            for j in range(N):
                acc += dS[i][j] * k[j][c]
            dQ[i][c] = scale * acc
    for j in range(N):
        for c in range(d):
            acc = 0.0
            for i in range(N):
                acc += dS[i][j] * q[i][c]
            dK[j][c] = scale * acc
    return dict(O=O, LSE=LSE, dQ=dQ, dK=dK, dV=dV)
