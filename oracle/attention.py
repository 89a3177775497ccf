"""CPU float64 oracle for exact scaled dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports or calls this module;
only the tests, the package's smoke check and the bench's CPU-baseline leg do.

What it computes is standard attention written out from its definition, with
S and P materialised (the pages' statement of the problem: S = Q K^T,
P = softmax(S), O = P V, with Q, K, V of N rows and d columns -- FlashAttention
milestone page (nlp-lineage), "The notation"). FlashAttention reaches this same
result exactly, only faster (FlashAttention proof-of-work page
(aiexpertsdirectory), FAQ "Is FlashAttention an approximation..."; Flash
Attention glossary (inferensys), paragraph on exactness), so the definition,
not the tiled algorithm, is the oracle. No blocking, online softmax or fusion
appears here.

Readings where the pages are silent (each also listed in the design notes):
  * scale is applied to the scores: S = scale * Q K^T.
  * Masks combine by AND: allowed(i, j) = (not causal or j <= i)
    and (j < kv_len[b]) and block_mask[i // 128, j // 128]; disallowed scores
    are -inf (the fused kernel's "mask" step, milestone page, "The idea").
  * LSE is the natural log-sum-exp of the scaled, masked scores, one per row
    (the "two numbers per row" kept for recomputation, milestone page,
    "The idea -- Recomputation", stored as m + ln l).
  * A row with no allowed key has O = 0, LSE = -inf and no gradient.
  * Backward (not written out on the pages; textbook softmax and matmul
    calculus for the loss L = sum(dO * O)):
        dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,
        dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
  * Tile states for a 128 x 128 grid: a tile is live when any of its elements
    (query row i < N) is allowed, and partial when it is live and some such
    element is not, keys past the end of the sequence counting as not
    allowed; 0 = skip, 1 = full, 2 = partial.

parity pins: see tests/test_oracle_pins.py (closed forms, brute force,
finite differences, an independent library routine).
"""
from __future__ import annotations

import numpy as np

TILE = 128
SKIP, FULL, PARTIAL = 0, 1, 2


def _f64(x):
    """Exact conversion of a (bf16/fp32 torch or numpy) array to float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _np(x, dtype):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").numpy().astype(dtype)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x).astype(dtype)


def allowed_mask(N, causal, kv_len_b=None, block_mask=None, tile=TILE):
    """Boolean [N, N] matrix of (query i, key j) pairs that take part.

    AND of the three masks the workloads use: causal (j <= i), key padding
    (j < kv_len_b) and a block mask over tile x tile blocks shared by all
    batches and heads (block-sparse FlashAttention skips the blocks a fixed
    sparsity pattern marks empty -- milestone page, "The idea").
    """
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    a = np.ones((N, N), dtype=bool)
    if causal:
        a &= j <= i
    if kv_len_b is not None:
        a &= j < int(kv_len_b)
    if block_mask is not None:
        bm = _np(block_mask, np.uint8).astype(bool)
        a &= bm[i // tile, j // tile]
    return a


def head_forward(q, k, v, scale, allowed):
    """Standard attention for one head, float64, S and P materialised.

    Returns dict(S=scaled masked scores, P, O, LSE).
    """
    S = scale * (q @ k.T)
    S = np.where(allowed, S, -np.inf)
    m = S.max(axis=1)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.exp(S - m_safe[:, None])           # exp(-inf) = 0 on masked pairs
    l = E.sum(axis=1)
    l_safe = np.where(empty, 1.0, l)
    P = E / l_safe[:, None]
    O = P @ v
    with np.errstate(divide="ignore"):
        LSE = np.where(empty, -np.inf, m_safe + np.log(l_safe))
    return dict(S=S, P=P, O=O, LSE=LSE)


def head_backward(q, k, v, do, scale, P, O):
    """Analytic gradient of L = sum(dO * O) for one head, float64."""
    dV = P.T @ do
    dP = do @ v.T
    D = (do * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return dict(dP=dP, D=D, dS=dS, dQ=dQ, dK=dK, dV=dV)


def head_rows(q, k, v, do, scale, causal, rows, keys, chunk=64):
    """Selected outputs of one head, float64, for lengths whose N x N matrices
    do not fit: O, LSE and dQ of the query rows ``rows``, dK and dV of the key
    rows ``keys``. The same definition as head_forward / head_backward,
    evaluated for blocks of query rows at a time (only the causal mask).

    A key's gradient sums over every query row that may attend to it: with
    causal masking those are the rows at or after the key, so keys near the
    end need few rows; without it every row is visited.
    Returns dict(O [len(rows), d], LSE [len(rows)], dQ [len(rows), d],
    dK [len(keys), d], dV [len(keys), d]).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    N, d = q.shape
    rows = [int(i) for i in rows]
    keys = [int(j) for j in keys]
    first = min(keys) if (keys and causal) else 0
    need = sorted(set(rows) | (set(range(first, N)) if keys else set()))
    pos = {i: n for n, i in enumerate(rows)}
    out = dict(O=np.zeros((len(rows), d)), LSE=np.zeros(len(rows)), dQ=np.zeros((len(rows), d)),
               dK=np.zeros((len(keys), d)), dV=np.zeros((len(keys), d)))
    kj = np.array(keys, dtype=np.int64)
    for c0 in range(0, len(need), chunk):
        I = np.array(need[c0:c0 + chunk], dtype=np.int64)
        allowed = (np.arange(N)[None, :] <= I[:, None]) if causal else np.ones((len(I), N), bool)
        f = head_forward(q[I], k, v, scale, allowed)
        g = head_backward(q[I], k, v, do[I], scale, f["P"], f["O"])
        for n, i in enumerate(I):
            if int(i) in pos:
                r = pos[int(i)]
                out["O"][r], out["LSE"][r], out["dQ"][r] = f["O"][n], f["LSE"][n], g["dQ"][n]
        if len(keys):
            out["dV"] += f["P"][:, kj].T @ do[I]
            out["dK"] += scale * (g["dS"][:, kj].T @ q[I])
    return out


def attention_fwd(q, k, v, scale, causal=False, kv_len=None, block_mask=None,
                  heads=None):
    """Batched forward on [B, H, N, d] inputs.

    Returns (O float64 [B, H, N, d], LSE float64 [B, H, N]). ``heads`` (a list
    of (b, h) pairs) restricts the work to those heads; the others stay NaN.
    """
    Q, K, V = _f64(q), _f64(k), _f64(v)
    B, H, N, d = Q.shape
    kvl = _np(kv_len, np.int64)
    O = np.full((B, H, N, d), np.nan)
    LSE = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    masks = {}
    for b, h in pairs:
        key = None if kvl is None else int(kvl[b])
        if key not in masks:
            masks[key] = allowed_mask(N, causal, key, block_mask)
        r = head_forward(Q[b, h], K[b, h], V[b, h], scale, masks[key])
        O[b, h], LSE[b, h] = r["O"], r["LSE"]
    return O, LSE


def attention_fwd_bwd(q, k, v, do, scale, causal=False, kv_len=None,
                      block_mask=None, heads=None):
    """Batched forward and backward on [B, H, N, d] inputs.

    Returns dict(O, LSE, D, dQ, dK, dV) in float64; heads outside ``heads``
    stay NaN.
    """
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, d = Q.shape
    kvl = _np(kv_len, np.int64)
    out = {n: np.full((B, H, N, d), np.nan) for n in ("O", "dQ", "dK", "dV")}
    out["LSE"] = np.full((B, H, N), np.nan)
    out["D"] = np.full((B, H, N), np.nan)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    masks = {}
    for b, h in pairs:
        key = None if kvl is None else int(kvl[b])
        if key not in masks:
            masks[key] = allowed_mask(N, causal, key, block_mask)
        f = head_forward(Q[b, h], K[b, h], V[b, h], scale, masks[key])
        g = head_backward(Q[b, h], K[b, h], V[b, h], dO[b, h], scale, f["P"], f["O"])
        out["O"][b, h], out["LSE"][b, h] = f["O"], f["LSE"]
        out["D"][b, h] = g["D"]
        out["dQ"][b, h], out["dK"][b, h], out["dV"][b, h] = g["dQ"], g["dK"], g["dV"]
        del f, g
    return out


def tile_states(B, N, causal, kv_len=None, block_mask=None, tile=TILE):
    """uint8 [B, nT, nT] tile states read off the element mask.

    The key axis is taken over the padded range [0, nT * tile), where keys
    j >= N never take part; only query rows i < N count (rows past the end of
    the sequence are not outputs). 0 = skip (no allowed element), 1 = full
    (every counted element allowed), 2 = partial (live, but some counted
    element disallowed).
    """
    nT = (N + tile - 1) // tile
    Np = nT * tile
    kvl = _np(kv_len, np.int64)
    out = np.zeros((B, nT, nT), dtype=np.uint8)
    for b in range(B):
        a = np.zeros((N, Np), dtype=bool)
        a[:, :N] = allowed_mask(N, causal, None if kvl is None else int(kvl[b]),
                                block_mask, tile)
        for qi in range(nT):
            for kj in range(nT):
                blk = a[qi * tile:(qi + 1) * tile, kj * tile:(kj + 1) * tile]
                if not blk.any():
                    out[b, qi, kj] = SKIP
                elif blk.all():
                    out[b, qi, kj] = FULL
                else:
                    out[b, qi, kj] = PARTIAL
    return out
