"""Pins for the CPU float64 oracle, against facts fixed outside the oracle.

Each test ties the oracle to a closed form, a brute-force or finite-difference
computation, an independent library routine (PyTorch's CPU scaled dot-product
attention and autograd), or hand-derived tile states, so that a dropped term,
a wrong sign or index, or a transposed operand anywhere in it fails one of
them. The last block plants such mistakes in copies of the oracle's gradient
and checks that the finite-difference pin catches each one.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

RNG = np.random.default_rng(1234)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


def _one_head(N, d, causal=False, kv=None, bm=None, seed=0, scale=None):
    rng = np.random.default_rng(seed)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    a = oa.allowed_mask(N, causal, kv, bm)
    f = oa.head_forward(q, k, v, scale, a)
    g = oa.head_backward(q, k, v, do, scale, f["P"], f["O"])
    return q, k, v, do, scale, a, f, g


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal,kv,bm", [
    (False, None, None), (True, None, None), (False, 200, None), (True, 150, None),
    (False, None, np.array([[1, 0, 1], [0, 1, 0], [1, 1, 1]], np.uint8)),
])
def test_zero_queries_give_mean_of_allowed_values(causal, kv, bm):
    """Q = 0 makes every allowed score 0, so P is uniform over the allowed
    keys: O_i is the mean of those V rows and LSE_i = ln(count_i)."""
    N, d = 300, 8
    k, v = _rand(N, d), _rand(N, d)
    q = np.zeros((N, d))
    a = oa.allowed_mask(N, causal, kv, bm)
    f = oa.head_forward(q, k, v, 0.37, a)
    for i in range(N):
        idx = np.nonzero(a[i])[0]
        if len(idx) == 0:
            assert f["LSE"][i] == -np.inf and np.all(f["O"][i] == 0)
            continue
        np.testing.assert_allclose(f["O"][i], v[idx].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(f["LSE"][i] - math.log(len(idx))) < 1e-13


def test_dominant_score_selects_one_value_row():
    """If Q_i = c K_j with c large, score j dominates and O_i -> V_j; the gap
    bounds the error by (N - 1) exp(-gap) max|V - V_j|."""
    N, d, scale = 64, 16, 0.25
    rng = np.random.default_rng(7)
    k = rng.standard_normal((N, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)     # unit keys
    v = rng.standard_normal((N, d))
    perm = rng.permutation(N)
    c = 200.0
    q = c * k[perm]
    f = oa.head_forward(q, k, v, scale, np.ones((N, N), bool))
    S = f["S"]
    for i in range(N):
        j = perm[i]
        gap = S[i, j] - np.max(np.delete(S[i], j))
        assert gap > 0
        bound = (N - 1) * math.exp(-gap) * 2 * np.abs(v).max() + 1e-14
        assert np.max(np.abs(f["O"][i] - v[j])) <= bound
        assert abs(f["LSE"][i] - S[i, j]) <= (N - 1) * math.exp(-gap) + 1e-14


def test_causal_row_zero_is_first_value_row():
    """Under the causal mask row 0 sees only key 0: O_0 = V_0 and
    LSE_0 = scale * q_0 . k_0 exactly."""
    q, k, v, do, scale, a, f, g = _one_head(50, 12, causal=True, seed=3)
    assert np.array_equal(f["O"][0], v[0])
    assert f["LSE"][0] == scale * (q[0] @ k[0])


def test_probability_rows_sum_to_one_and_dS_rows_to_zero():
    """Softmax rows sum to 1; every row of dS sums to 0 because
    D_i = sum_j P_ij dP_ij."""
    for causal, kv in [(False, None), (True, None), (False, 70)]:
        *_, f, g = _one_head(150, 16, causal=causal, kv=kv, seed=5)
        np.testing.assert_allclose(f["P"].sum(axis=1), 1.0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(g["dS"].sum(axis=1), 0.0, rtol=0, atol=1e-11)
        assert np.all(f["P"][~oa.allowed_mask(150, causal, kv)] == 0)


def test_fully_masked_rows_are_zero_with_minus_inf_lse():
    q, k, v, do, scale, a, f, g = _one_head(20, 4, kv=0, seed=9)
    assert np.all(f["O"] == 0) and np.all(f["LSE"] == -np.inf)
    assert np.all(g["dQ"] == 0) and np.all(g["dK"] == 0) and np.all(g["dV"] == 0)


# --------------------------------------------------------------------------
# Brute force and finite differences
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal,kv,bm,tile", [
    (False, None, None, 128), (True, None, None, 128), (False, 9, None, 128),
    (True, 11, None, 128),
    (False, None, [[1, 0, 1, 1], [0, 1, 0, 0], [1, 1, 1, 0], [0, 0, 1, 1]], 4),
    (True, 14, [[1, 0, 0, 0], [1, 1, 0, 0], [0, 1, 1, 0], [1, 0, 1, 1]], 4),
])
def test_numpy_oracle_matches_scalar_loops(causal, kv, bm, tile):
    N, d = 16, 5
    rng = np.random.default_rng(11)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    scale = 0.45
    bm_np = None if bm is None else np.array(bm, np.uint8)
    a = oa.allowed_mask(N, causal, kv, bm_np, tile=tile)
    f = oa.head_forward(q, k, v, scale, a)
    g = oa.head_backward(q, k, v, do, scale, f["P"], f["O"])
    ref = oracle.loop_attention_fwd_bwd(q.tolist(), k.tolist(), v.tolist(), do.tolist(),
                                        scale, causal, kv, bm, tile)
    np.testing.assert_allclose(f["O"], ref["O"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(f["LSE"], ref["LSE"], rtol=0, atol=1e-13)
    for n in ("dQ", "dK", "dV"):
        np.testing.assert_allclose(g[n], ref[n], rtol=0, atol=1e-12)


def _loss(q, k, v, do, scale, a):
    return float((oa.head_forward(q, k, v, scale, a)["O"] * do).sum())


def _fd_grads(q, k, v, do, scale, a, h=1e-6):
    out = []
    for which in range(3):
        xs = [q.copy(), k.copy(), v.copy()]
        grad = np.zeros_like(xs[which])
        for idx in np.ndindex(grad.shape):
            xp = [x.copy() for x in xs]
            xm = [x.copy() for x in xs]
            xp[which][idx] += h
            xm[which][idx] -= h
            grad[idx] = (_loss(*xp, do, scale, a) - _loss(*xm, do, scale, a)) / (2 * h)
        out.append(grad)
    return out


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, 5), (True, 6)])
def test_backward_matches_finite_differences(causal, kv):
    N, d = 8, 4
    q, k, v, do, scale, a, f, g = _one_head(N, d, causal=causal, kv=kv, seed=21, scale=0.8)
    fdq, fdk, fdv = _fd_grads(q, k, v, do, scale, a)
    assert _rel(g["dQ"], fdq) < 1e-7
    assert _rel(g["dK"], fdk) < 1e-7
    assert _rel(g["dV"], fdv) < 1e-7


# --------------------------------------------------------------------------
# Independent library routine: PyTorch CPU scaled dot-product attention
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal,use_kv,use_bm", [
    (False, False, False), (True, False, False), (False, True, False),
    (False, False, True), (True, True, True),
])
def test_matches_torch_sdpa_and_autograd_in_float64(causal, use_kv, use_bm):
    B, H, N, d = 2, 2, 300, 16
    g = torch.Generator().manual_seed(4)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g, dtype=torch.float64) for _ in range(4))
    kv = torch.tensor([260, 131], dtype=torch.int32) if use_kv else None
    nT = 3
    bm = torch.tensor([[1, 0, 1], [1, 1, 0], [0, 1, 1]], dtype=torch.uint8) if use_bm else None
    scale = 0.3
    ref = oa.attention_fwd_bwd(q, k, v, do, scale, causal, kv, bm)
    # the same mask, built independently of the oracle: causal via triu,
    # padding via a key-index comparison, blocks via a Kronecker expansion
    mask = torch.ones(B, 1, N, N, dtype=torch.bool)
    if causal:
        mask &= ~torch.triu(torch.ones(N, N, dtype=torch.bool), diagonal=1)
    if kv is not None:
        mask &= (torch.arange(N)[None, :] < kv[:, None].long())[:, None, None, :]
    if bm is not None:
        mask &= torch.kron(bm, torch.ones(128, 128, dtype=torch.uint8))[:N, :N].bool()
    assert mask.any(dim=-1).all(), "test case must not have fully masked rows"
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
    o.backward(do)
    np.testing.assert_allclose(ref["O"], o.detach().numpy(), rtol=0, atol=1e-12)
    for n, t in (("dQ", qq), ("dK", kk), ("dV", vv)):
        np.testing.assert_allclose(ref[n], t.grad.numpy(), rtol=0, atol=1e-11)
    s = scale * (q @ k.transpose(-1, -2))
    s = s.masked_fill(~mask, -math.inf)
    np.testing.assert_allclose(ref["LSE"], torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_block_sparse_equals_dense_with_minus_inf_blocks():
    """Block-sparse attention for a fixed block mask is dense attention with
    the masked blocks' scores set to -inf (the mask built here by expanding
    the blocks element by element, not by the oracle's index arithmetic)."""
    N, d = 512, 8
    rng = np.random.default_rng(2)
    bm = (rng.random((4, 4)) < 0.4).astype(np.uint8)
    np.fill_diagonal(bm, 1)
    q, k, v = _rand(N, d), _rand(N, d), _rand(N, d)
    sparse = oa.head_forward(q, k, v, 0.5, oa.allowed_mask(N, False, None, bm))
    S = 0.5 * q @ k.T
    for bi in range(4):
        for bj in range(4):
            if not bm[bi, bj]:
                S[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128] = -np.inf
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    P /= P.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(sparse["O"], P @ v, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# The tiled online-softmax reading of the method equals the oracle
# --------------------------------------------------------------------------

def _online_softmax_model(q, k, v, scale, a, Br, Bc, tau):
    """Float64 model of the tiled forward as read from the pages: for each
    block of Br query rows, stream blocks of Bc keys, keep a running row max
    m and row sum l, rescale the earlier partial output when m grows
    (FlashAttention milestone page (nlp-lineage), "The idea -- Tiling";
    pixelation.org article, "The Online Softmax Trick"). The reference max
    is only moved when the new max exceeds it by more than tau (tau = 0
    moves it every time); the result is the same for any tau."""
    N, d = q.shape
    O = np.zeros((N, d))
    LSE = np.zeros(N)
    for r0 in range(0, N, Br):
        rows = slice(r0, min(N, r0 + Br))
        nr = rows.stop - rows.start
        m = np.full(nr, -np.inf)
        l = np.zeros(nr)
        acc = np.zeros((nr, d))
        for c0 in range(0, N, Bc):
            cols = slice(c0, min(N, c0 + Bc))
            s = scale * q[rows] @ k[cols].T
            s = np.where(a[rows, cols], s, -np.inf)
            mt = s.max(axis=1)
            move = mt > m + tau
            m_new = np.where(move, mt, m)
            alpha = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(m_new), m_new, 0)), 0.0)
            alpha = np.where(move, alpha, 1.0)
            ref = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.exp(s - ref[:, None])
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ v[cols]
            m = m_new
        empty = l == 0
        O[rows] = np.where(empty[:, None], 0.0, acc / np.where(empty, 1, l)[:, None])
        with np.errstate(divide="ignore"):
            LSE[rows] = np.where(empty, -np.inf, np.where(np.isfinite(m), m, 0) + np.log(np.where(empty, 1, l)))
    return O, LSE


@pytest.mark.parametrize("tau", [0.0, 8.0 * math.log(2.0)])
@pytest.mark.parametrize("causal,kv", [(False, None), (True, None), (False, 333)])
def test_tiled_online_softmax_equals_oracle(causal, kv, tau):
    N, d = 500, 16
    q, k, v, do, scale, a, f, g = _one_head(N, d, causal=causal, kv=kv, seed=31)
    O, LSE = _online_softmax_model(q, k, v, scale, a, 128, 128, tau)
    np.testing.assert_allclose(O, f["O"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, f["LSE"], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Tile states against hand-derived fixtures
# --------------------------------------------------------------------------

def _parse_golden(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(" ")
        if key == "case":
            cur = dict(name=val, rows={})
        elif key == "end":
            cases.append(cur)
        elif key in ("N", "causal"):
            cur[key] = int(val)
        elif key == "kv_len":
            cur[key] = None if val == "-" else [int(x) for x in val.split(",")]
        elif key == "block_mask":
            cur[key] = None if val == "-" else [[int(x) for x in r.split(",")] for r in val.split("/")]
        elif key.startswith("b"):
            cur["rows"][int(key[1:])] = [[int(x) for x in r.split(",")] for r in val.split("/")]
    return cases


@pytest.mark.parametrize("case", _parse_golden(os.path.join(GOLDEN, "tile_states.txt")),
                         ids=lambda c: c["name"])
def test_tile_states_match_hand_derived(case):
    B = len(case["rows"])
    kv = None if case["kv_len"] is None else np.array(case["kv_len"])
    bm = None if case["block_mask"] is None else np.array(case["block_mask"], np.uint8)
    got = oa.tile_states(B, case["N"], bool(case["causal"]), kv, bm)
    want = np.array([case["rows"][b] for b in range(B)], np.uint8)
    assert np.array_equal(got, want), (got, want)


# --------------------------------------------------------------------------
# Planted mistakes: each must be caught by the finite-difference pin
# --------------------------------------------------------------------------

def _bwd_dropped_scale(q, k, v, do, scale, P, O):
    r = oa.head_backward(q, k, v, do, scale, P, O)
    r["dQ"] = r["dQ"] / scale
    return r


def _bwd_wrong_sign(q, k, v, do, scale, P, O):
    dP = do @ v.T
    D = (do * O).sum(axis=1)
    dS = P * (dP + D[:, None])
    return dict(dQ=scale * dS @ k, dK=scale * dS.T @ q, dV=P.T @ do)


def _bwd_transposed(q, k, v, do, scale, P, O):
    r = oa.head_backward(q, k, v, do, scale, P, O)
    r["dV"] = P @ do
    return r


@pytest.mark.parametrize("bad", [_bwd_dropped_scale, _bwd_wrong_sign, _bwd_transposed])
def test_planted_gradient_mistakes_are_caught(bad):
    N, d = 8, 4
    q, k, v, do, scale, a, f, g = _one_head(N, d, causal=True, seed=21, scale=0.8)
    fdq, fdk, fdv = _fd_grads(q, k, v, do, scale, a)
    r = bad(q, k, v, do, scale, f["P"], f["O"])
    worst = max(_rel(r["dQ"], fdq), _rel(r["dK"], fdk), _rel(r["dV"], fdv))
    assert worst > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_the_full_oracle(causal):
    """head_rows (used where the N x N matrices do not fit) against the full
    oracle on a length that fits: the same values to rounding."""
    from oracle import attention as oa
    rng = np.random.default_rng(21)
    N, d, scale = 300, 16, 0.3
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    ref = oa.attention_fwd_bwd(q[None, None], k[None, None], v[None, None], do[None, None], scale, causal)
    rows, keys = [0, 1, 129, 250, 299], [299, 290, 200]
    got = oa.head_rows(q, k, v, do, scale, causal, rows, keys)
    for name, idx in (("O", rows), ("LSE", rows), ("dQ", rows), ("dK", keys), ("dV", keys)):
        np.testing.assert_allclose(got[name], ref[name][0, 0][idx], rtol=1e-12, atol=1e-12, err_msg=name)
