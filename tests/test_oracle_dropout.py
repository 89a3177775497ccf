"""Pins for the oracle's dropout: the counter-based generator, the keep mask,
and attention with dropout on P.

The generator is checked against a second, scalar spelling of Philox4x32-10
and against the statistics any good generator must show; the attention with
dropout against the undropped oracle at p = 0, finite differences under a
fixed mask, and unbiasedness over many seeds.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as oa
from oracle import dropout as od


def _kat_vectors():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    rows = []
    for line in open(path):
        line = line.split("#")[0].split()
        if line:
            w = [int(x, 16) for x in line]
            rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_generator_matches_published_known_answers():
    """Both spellings of the generator reproduce the published known-answer
    vectors of Philox4x32-10 (Random123), so a mistake shared by the two
    spellings (a wrong multiplier, Weyl constant or word order) would fail."""
    rows = _kat_vectors()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert od.philox4x32_10_scalar(ctr, key) == want
        got = [int(x) for x in od.philox4x32_10(*ctr, *key)]
        assert got == want


def test_vectorised_generator_matches_scalar_spelling():
    rng = np.random.default_rng(0)
    for _ in range(200):
        ctr = rng.integers(0, 2**32, size=4, dtype=np.uint64)
        key = rng.integers(0, 2**32, size=2, dtype=np.uint64)
        got = [int(x) for x in od.philox4x32_10(*ctr, *key)]
        assert got == od.philox4x32_10_scalar(ctr, key)


def test_generator_output_bytes_are_uniform_and_counters_decorrelate():
    n = 1 << 15
    c0 = np.arange(n, dtype=np.uint64)
    words = np.stack(od.philox4x32_10(c0, 7, 3, 0, 12345, 678))       # [4, n]
    b = words.view(np.uint8).reshape(-1)
    counts = np.bincount(b, minlength=256)
    expected = b.size / 256
    chi2 = ((counts - expected) ** 2 / expected).sum()
    # 255 degrees of freedom: mean 255, sd ~22.6; a 6-sd band
    assert abs(chi2 - 255) < 6 * math.sqrt(2 * 255)
    # neighbouring counters give unrelated words: bit agreement near 1/2
    x = words[0]
    agree = np.unpackbits((~(x[:-1] ^ x[1:])).view(np.uint8)).mean()
    assert abs(agree - 0.5) < 0.01


@pytest.mark.parametrize("p", [0.1, 0.25, 0.5, 0.9])
def test_keep_fraction_matches_threshold(p):
    N = 512
    keep, s = od.keep_mask(seed=99, bh=5, N=N, p_drop=p)
    t, s2 = od.threshold(p)
    q = (256 - t) / 256
    frac = keep.mean()
    sd = math.sqrt(q * (1 - q) / keep.size)
    assert abs(frac - q) < 6 * sd
    assert s == s2 == 256.0 / (256 - t)


def test_mask_layout_against_scalar_calls():
    """Element (i, j) of head bh takes byte 4 (i mod 4) + (j mod 4) of the call
    with counter (i div 4, j div 4, bh, 0) and key (seed lo, seed hi)."""
    seed, bh, N = (0xDEADBEEF << 32) | 0x12345678, 11, 37
    rb = od.random_bytes(seed, bh, N)
    rng = np.random.default_rng(3)
    for _ in range(60):
        i, j = (int(x) for x in rng.integers(0, N, size=2))
        w = od.philox4x32_10_scalar((i // 4, j // 4, bh, 0), (seed & 0xFFFFFFFF, seed >> 32))
        assert rb[i, j] == (w[i % 4] >> (8 * (j % 4))) & 0xFF


def test_zero_probability_is_plain_attention():
    rng = np.random.default_rng(1)
    B, H, N, d = 1, 2, 200, 8
    q, k, v, do = (rng.standard_normal((B, H, N, d)) for _ in range(4))
    a = oa.attention_fwd_bwd(q, k, v, do, 0.4, True)
    b = od.attention_fwd_bwd_dropout(q, k, v, do, 0.4, True, p_drop=0.0, seed=5)
    for n in ("O", "LSE", "dQ", "dK", "dV"):
        np.testing.assert_array_equal(a[n], b[n])


def _loss(q, k, v, do, scale, allowed, keep, s):
    return float((od.head_forward_dropout(q, k, v, scale, allowed, keep, s)["O"] * do).sum())


def _fd(q, k, v, do, scale, allowed, keep, s, h=1e-6):
    out = []
    for which in range(3):
        xs = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(xs[which])
        for idx in np.ndindex(g.shape):
            xp = [x.copy() for x in xs]
            xm = [x.copy() for x in xs]
            xp[which][idx] += h
            xm[which][idx] -= h
            g[idx] = (_loss(*xp, do, scale, allowed, keep, s) - _loss(*xm, do, scale, allowed, keep, s)) / (2 * h)
        out.append(g)
    return out


def _rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_backward_matches_finite_differences(causal):
    N, d, scale = 8, 4, 0.7
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    allowed = oa.allowed_mask(N, causal)
    keep, s = od.keep_mask(seed=4, bh=0, N=N, p_drop=0.3)
    assert 0 < keep.mean() < 1
    f = od.head_forward_dropout(q, k, v, scale, allowed, keep, s)
    g = od.head_backward_dropout(q, k, v, do, scale, f["P"], f["Pd"], f["O"], keep, s)
    fq, fk, fv = _fd(q, k, v, do, scale, allowed, keep, s)
    assert _rel(g["dQ"], fq) < 1e-7 and _rel(g["dK"], fk) < 1e-7 and _rel(g["dV"], fv) < 1e-7


def test_planted_dropout_mistake_is_caught():
    """Forgetting the mask and scale on dP breaks the finite-difference pin."""
    N, d, scale = 8, 4, 0.7
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((N, d)) for _ in range(4))
    allowed = oa.allowed_mask(N, False)
    keep, s = od.keep_mask(seed=4, bh=0, N=N, p_drop=0.3)
    f = od.head_forward_dropout(q, k, v, scale, allowed, keep, s)
    bad = od.head_backward_dropout(q, k, v, do, scale, f["P"], f["Pd"], f["O"], np.ones_like(keep), 1.0)
    fq, _, _ = _fd(q, k, v, do, scale, allowed, keep, s)
    assert _rel(bad["dQ"], fq) > 1e-3


def test_dropout_is_unbiased_over_seeds():
    """E[O] over seeds equals the undropped output (scale 256 / (256 - t))."""
    N, d, scale = 16, 4, 0.5
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    allowed = oa.allowed_mask(N, False)
    ref = oa.head_forward(q, k, v, scale, allowed)["O"]
    acc = np.zeros_like(ref)
    n = 4000
    for seed in range(n):
        keep, s = od.keep_mask(seed, 0, N, 0.5)
        acc += od.head_forward_dropout(q, k, v, scale, allowed, keep, s)["O"]
    # per-element standard error of the mean is below ~0.02 here
    assert np.abs(acc / n - ref).max() < 0.1
