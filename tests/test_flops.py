"""FLOP accounting (host logic) against the oracle's element mask."""
import numpy as np
import pytest

import oracle
from exact_io_aware_39_gb300.flops import allowed_pairs, attention_flops


@pytest.mark.parametrize("N,causal,kv,bm", [
    (256, False, None, None), (300, True, None, None), (384, False, [200, 384, 0, 128], None),
    (384, True, [130, 1], None),
    (384, False, None, [[1, 0, 1], [0, 1, 0], [1, 1, 1]]),
    (384, True, [300], [[1, 0, 0], [1, 0, 0], [0, 1, 1]]),
])
def test_allowed_pairs_match_element_mask(N, causal, kv, bm):
    B = 1 if kv is None else len(kv)
    bm_np = None if bm is None else np.array(bm, np.uint8)
    got = allowed_pairs(B, N, causal, kv, bm_np)
    for b in range(B):
        a = oracle.allowed_mask(N, causal, None if kv is None else kv[b], bm_np)
        assert got[b] == a.sum()


def test_flops_closed_forms():
    f, b = attention_flops(1, 2, 256, 64, False)
    assert f == 4 * 64 * 256 * 256 * 2 and b == 2.5 * f
    N = 1024
    f, _ = attention_flops(8, 16, N, 64, True)
    assert f == 4 * 64 * (N * (N + 1) // 2) * 8 * 16
