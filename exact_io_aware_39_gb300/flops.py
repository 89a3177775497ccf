"""Algorithmic work of exact attention, counted over the (query, key) pairs
that take part (allowed by the causal, key-length and block masks).

Per allowed pair and head dimension d the forward pass does two
multiply-adds per column (one in S = Q K^T, one in O = P V): 4 d FLOP. The
backward pass does five such products (S recomputed, dP, dV, dK, dQ):
10 d FLOP, i.e. 2.5 times the forward. Masked pairs inside computed tiles
and skipped tiles are not counted.
"""
from __future__ import annotations

import numpy as np

TILE = 128


def allowed_pairs(B, N, causal, kv_len=None, block_mask=None):
    """Number of allowed (i, j) pairs per batch entry, as an int64 array [B].

    Counted tile by tile in closed form: in tile (qi, kj), row i sees the keys
    j in [128 kj, hi) with hi = min(128 kj + 128, kv_len, i + 1 if causal).
    """
    nT = (N + TILE - 1) // TILE
    kvl = np.full(B, N, dtype=np.int64) if kv_len is None else np.clip(
        np.asarray(kv_len, dtype=np.int64).reshape(-1), 0, N)
    bm = None if block_mask is None else np.asarray(block_mask).astype(bool)
    rows = np.arange(N, dtype=np.int64)
    out = np.zeros(B, dtype=np.int64)
    for b in range(B):
        total = 0
        for kj in range(nT):
            lo = kj * TILE
            hi = np.minimum(lo + TILE, kvl[b])
            if hi <= lo:
                continue
            if bm is None:
                r = rows
            else:
                live_q = np.repeat(bm[:, kj], TILE)[:N]
                r = rows[live_q]
            lim = np.minimum(hi, r + 1) if causal else np.full(r.shape, hi)
            total += int(np.maximum(lim - lo, 0).sum())
        out[b] = total
    return out


def attention_flops(B, H, N, d, causal, kv_len=None, block_mask=None):
    """(forward FLOP, backward FLOP) of one call."""
    pairs = int(allowed_pairs(B, N, causal, kv_len, block_mask).sum()) * H
    fwd = 4 * d * pairs
    return fwd, 2.5 * fwd
