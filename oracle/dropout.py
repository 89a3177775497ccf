"""Dropout on P for the CPU oracle: counter-based random numbers and the keep mask.

TEST INFRASTRUCTURE ONLY (like the rest of this package).

The fused kernel of the method applies dropout to P between the two matrix
products and regenerates the same mask in the backward pass instead of storing
it (FlashAttention milestone page (nlp-lineage), "The idea": matrix multiply,
mask, softmax, dropout, matrix multiply in one kernel; Flash Attention
glossary, kernel-fusion paragraph). The pages name no generator, so both the
oracle and the CUDA path use Philox4x32-10 (Salmon, Moraes, Dror and Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011), each written
independently from that published definition:

  state: counter (c0, c1, c2, c3), key (k0, k1), 32-bit words;
  round: (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2 (64-bit products),
         c <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0);
  ten rounds; before every round but the first the key grows by
  (W0, W1) modulo 2^32.
  M0 = 0xD2511F53, M1 = 0xCD9E8D57, W0 = 0x9E3779B9, W1 = 0xBB67AE85.

Mask (the reading used here, stated in the design notes): for batch b, head
h (bh = b * H + h), query i and key j, one generator call with key
(seed mod 2^32, seed div 2^32) and counter (i div 4, j div 4, bh, 0) yields 16
bytes, little-endian across the four output words; element (i, j) takes byte
4 * (i mod 4) + (j mod 4). It is kept when that byte is >= t, with
t = round(256 p) (so p is used in steps of 1/256), and a kept element is
scaled by 256 / (256 - t), which keeps O unbiased.
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10 on uint32 arrays (broadcast together).
    Returns the four output words as uint32 arrays."""
    c0, c1, c2, c3 = (np.asarray(x, dtype=np.uint64) & MASK32 for x in (c0, c1, c2, c3))
    k0 = np.asarray(k0, dtype=np.uint64) & MASK32
    k1 = np.asarray(k1, dtype=np.uint64) & MASK32
    for r in range(10):
        if r > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = np.uint64(M0) * c0            # < 2^64, exact in uint64
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ k0), lo1, (hi0 ^ c3 ^ k1), lo0
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def philox4x32_10_scalar(ctr, key):
    """Plain-integer spelling of the same generator (a pin for the vectorised
    one on small inputs)."""
    c = [int(x) & MASK32 for x in ctr]
    k = [int(x) & MASK32 for x in key]
    for r in range(10):
        if r > 0:
            k = [(k[0] + W0) & MASK32, (k[1] + W1) & MASK32]
        a = M0 * c[0]
        b = M1 * c[2]
        c = [((b >> 32) ^ c[1] ^ k[0]) & MASK32, b & MASK32, ((a >> 32) ^ c[3] ^ k[1]) & MASK32, a & MASK32]
    return c


def threshold(p_drop):
    """Integer threshold t of the byte test and the scale 256 / (256 - t)."""
    if not (0.0 <= p_drop < 1.0):
        raise ValueError("p_drop must be in [0, 1)")
    t = int(np.floor(p_drop * 256.0 + 0.5))
    if t > 255:
        raise ValueError("p_drop rounds to 256/256")
    return t, 256.0 / (256.0 - t)


def random_bytes(seed, bh, N):
    """uint8 [N, N] byte of every (query i, key j) pair of head bh."""
    nb = (N + 3) // 4
    ib = np.arange(nb, dtype=np.uint64)[:, None]
    jb = np.arange(nb, dtype=np.uint64)[None, :]
    words = philox4x32_10(ib, jb, bh, 0, seed & MASK32, (seed >> 32) & MASK32)   # each [nb, nb]
    out = np.empty((nb * 4, nb * 4), dtype=np.uint8)
    for r in range(4):                          # query i mod 4 -> word r
        w = words[r]
        for c in range(4):                      # key j mod 4 -> byte c of the word
            out[r::4, c::4] = ((w >> np.uint32(8 * c)) & np.uint32(0xFF)).astype(np.uint8)
    return out[:N, :N]


def keep_mask(seed, bh, N, p_drop):
    """bool [N, N] keep decisions of head bh, and the scale of kept values."""
    t, s = threshold(p_drop)
    return random_bytes(seed, bh, N) >= t, s


def head_forward_dropout(q, k, v, scale, allowed, keep, keep_scale):
    """One head: softmax statistics from the undropped P; O from the dropped P."""
    from .attention import head_forward
    f = head_forward(q, k, v, scale, allowed)
    Pd = f["P"] * keep * keep_scale
    f["Pd"] = Pd
    f["O"] = Pd @ v
    return f


def head_backward_dropout(q, k, v, do, scale, P, Pd, O, keep, keep_scale):
    """Gradient of L = sum(dO * O) with O = (P * Z * s) V:
    dV = Pd^T dO, dP = (dO V^T) * Z * s, D = rowsum(dO * O), dS = P * (dP - D)."""
    dV = Pd.T @ do
    dP = (do @ v.T) * keep * keep_scale
    D = (do * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    return dict(dP=dP, D=D, dS=dS, dQ=scale * (dS @ k), dK=scale * (dS.T @ q), dV=dV)


def attention_fwd_bwd_dropout(q, k, v, do, scale, causal=False, kv_len=None, block_mask=None,
                              p_drop=0.0, seed=0, heads=None):
    """Batched forward and backward with dropout on P, float64."""
    from .attention import _f64, _np, allowed_mask
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = Q.shape
    kvl = _np(kv_len, np.int64)
    out = {n: np.full((B, H, N, d), np.nan) for n in ("O", "dQ", "dK", "dV")}
    out["LSE"] = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        a = allowed_mask(N, causal, None if kvl is None else int(kvl[b]), block_mask)
        keep, s = keep_mask(seed, b * H + h, N, p_drop)
        f = head_forward_dropout(Q[b, h], K[b, h], V[b, h], scale, a, keep, s)
        g = head_backward_dropout(Q[b, h], K[b, h], V[b, h], dO[b, h], scale, f["P"], f["Pd"], f["O"], keep, s)
        out["O"][b, h], out["LSE"][b, h] = f["O"], f["LSE"]
        out["dQ"][b, h], out["dK"][b, h], out["dV"][b, h] = g["dQ"], g["dK"], g["dV"]
    return out
