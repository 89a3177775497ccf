"""GPU parity of dropout on P (fa_options.p_drop, fa_options.seed) against the
oracle's dropout, and bit-exact keep masks from both kernels' generators.

Tolerances as for the other parity tests (LSE max-abs <= 1e-3, dQ/dK/dV
relative Frobenius <= 2e-2), except O: dropout multiplies the kept values by
s = 256 / (256 - t), so O can reach s times the magnitudes of the undropped
case, and rounding O to bf16 (8 significant bits) alone moves an element by
up to 2^-8 |O| (0.016 at |O| = 4.1, 0.035 at |O| = 9 in early causal rows at
p = 0.5). P itself enters the P V product in the 16-bit input format (the
format the pages name for the tensor-core products: glossary page, "Tensor
Cores"; article, "Actionable Next Steps"), half an ulp of relative error per
term, so O moves by up to 2^-9 * s * sum_j P_j |V_j| <= 2^-9 * s * max |V| of
the head (the P of a row sums to at most 1). The O bound is therefore
elementwise 1e-2 * s + 2^-8 |O_ref| + 2^-9 * s * max |V|. The keep masks are
compared bit for bit.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_39_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

O_TOL, LSE_TOL, GRAD_TOL = 1e-2, 1e-3, 2e-2


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_39_gb300 as pkg
    from exact_io_aware_39_gb300 import build as b
    pkg.load(b.build())
    return pkg


CASES = [
    # name, B, H, N, d, causal, kv_len, block mask, p, seed, dtype
    ("d64_plain", 1, 2, 256, 64, False, None, False, 0.1, 7, torch.bfloat16),
    ("d64_causal_ragged", 2, 2, 333, 64, True, None, False, 0.3, 1234, torch.bfloat16),
    ("d128_causal", 1, 3, 520, 128, True, None, False, 0.5, 99, torch.bfloat16),
    ("d64_kv_len", 3, 2, 300, 64, False, [300, 5, 130], False, 0.25, 2**40 + 3, torch.bfloat16),
    ("d128_block_mask", 1, 2, 640, 128, True, None, True, 0.2, 5, torch.bfloat16),
    ("fp16_d128", 1, 2, 384, 128, False, None, False, 0.3, 42, torch.float16),
    ("d80_causal", 1, 2, 300, 80, True, None, False, 0.2, 77, torch.bfloat16),
    # more (key tile, batch-head) items than twice the SMs of a GB300 (152), so
    # that the persistent backward kernel walks several items per CTA
    ("d64_many_items_kv_len", 4, 21, 512, 64, True, [512, 0, 300, 129], False, 0.2, 11, torch.bfloat16),
    ("d128_many_items", 2, 56, 384, 128, True, None, False, 0.1, 2**33 + 1, torch.bfloat16),
    ("fp16_d64_many_items_kv_len", 4, 21, 512, 64, False, [512, 200, 0, 384], False, 0.15, 3, torch.float16),
]


def _case(name, B, H, N, d, causal, kv, use_bm, p, seed, dtype):
    w = Workload(name, B, H, N, d, causal, 1.0 / math.sqrt(d))
    c = make_case(w, seed=zlib.crc32(name.encode()) % 1000, dtype=dtype)
    if kv is not None:
        c["kv_len"] = torch.tensor(kv, dtype=torch.int32)
    if use_bm:
        nT = (N + 127) // 128
        g = torch.Generator().manual_seed(5)
        m = (torch.rand(nT, nT, generator=g) < 0.5).to(torch.uint8)
        m[torch.arange(nT), torch.arange(nT)] = 1
        c["block_mask"] = m
    return c


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_dropout_matches_oracle(fa, spec):
    c = _case(*spec)
    p, seed = spec[8], spec[9]
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
    bm = None if c["block_mask"] is None else c["block_mask"].to(dev)
    o, lse = fa.attention_fwd(q, k, v, c["scale"], c["causal"], kv, bm, p_drop=p, seed=seed)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, c["scale"], c["causal"], kv, bm, p_drop=p, seed=seed)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    ref = oracle.attention_fwd_bwd_dropout(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"],
                                           c["kv_len"], c["block_mask"], p_drop=p, seed=seed)
    o_abs = np.abs(o.float().cpu().numpy() - ref["O"])
    keep_scale = oracle.threshold(p)[1]
    v_max = np.abs(c["v"].float().numpy()).max(axis=(2, 3), keepdims=True)   # per head
    bound = O_TOL * keep_scale + 2.0 ** -8 * np.abs(ref["O"]) + 2.0 ** -9 * keep_scale * v_max
    assert (o_abs <= bound).all(), (o_abs.max(), (o_abs - bound).max())
    lr, lg = ref["LSE"], lse.cpu().numpy()
    fin = np.isfinite(lr)
    assert np.array_equal(fin, np.isfinite(lg))
    assert np.abs(lg[fin] - lr[fin]).max() <= LSE_TOL
    for name, g in (("dQ", dq), ("dK", dk), ("dV", dv)):
        a = g.float().cpu().numpy()
        rel = np.linalg.norm(a - ref[name]) / np.linalg.norm(ref[name])
        assert rel <= GRAD_TOL, (name, rel)


@pytest.mark.parametrize("p,seed", [(0.3, 17), (0.7, (5 << 32) | 9)])
def test_dropout_masks_bit_exact(fa, p, seed):
    """Q = 0 makes P uniform (1/N); with V_j = w_j e_(j mod 128), w = 1 for
    the first 128 keys and 2 for the next, each forward output element
    O[i, c] = (Z[i, c] + 2 Z[i, c + 128]) s / N reveals two keep bits. In the
    backward pass dO = I on the first 128 queries gives dV[j, c] =
    Z[c, j] s / N for keys j: the transposed mask from the other generator
    path."""
    B, H, N, d = 1, 2, 256, 128
    dev = torch.device("cuda:0")
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device=dev)
    k = torch.randn(B, H, N, d, dtype=torch.bfloat16, device=dev)
    eye = torch.eye(128)
    v = torch.cat([eye, 2 * eye], 0).to(torch.bfloat16)[None, None].repeat(B, H, 1, 1).to(dev)
    o, lse = fa.attention_fwd(q, k, v, 1.0, False, p_drop=p, seed=seed)
    do = torch.cat([eye, torch.zeros(128, 128)], 0).to(torch.bfloat16)[None, None].repeat(B, H, 1, 1).to(dev)
    dq, dk, dv = fa.attention_bwd(q, k, v, o, do, lse, 1.0, False, p_drop=p, seed=seed)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    t, s = oracle.threshold(p)
    unit = s / N
    for h in range(H):
        keep, _ = oracle.keep_mask(seed, h, N, p)
        code = np.rint(o[0, h].float().cpu().numpy() / unit).astype(np.int64)     # [N, 128]
        want = keep[:, :128].astype(np.int64) + 2 * keep[:, 128:].astype(np.int64)
        assert np.array_equal(code, want), f"forward mask differs for head {h}"
        got_t = np.rint(dv[0, h].float().cpu().numpy() / unit).astype(np.int64)   # [keys, 128 queries]
        assert np.array_equal(got_t, keep[:128, :].T.astype(np.int64)), f"backward mask differs for head {h}"


@pytest.mark.parametrize("p,seed", [(0.3, 23), (0.6, (3 << 32) | 5)])
def test_dropout_masks_bit_exact_d64(fa, p, seed):
    """The same at d = 64 (the 64-column kernels: their forward, and the
    backward's four P/dS warpgroups of 32 queries). With 64 value columns
    V_j = w_j e_(j mod 64) carries four keys per column, w = 1, 2, 4, 8 for
    keys 0-63, 64-127, 128-191, 192-255, so O[i, c] = (Z[i, c] + 2 Z[i, c + 64]
    + 4 Z[i, c + 128] + 8 Z[i, c + 192]) s / N, a 4-bit code. In the backward
    pass dO = I on queries 64 m .. 64 m + 63 gives dV[j, c] = Z[64 m + c, j] s / N;
    two calls cover the first query tile."""
    B, H, N, d = 1, 2, 256, 64
    dev = torch.device("cuda:0")
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device=dev)
    k = torch.randn(B, H, N, d, dtype=torch.bfloat16, device=dev)
    eye = torch.eye(64)
    v = torch.cat([eye, 2 * eye, 4 * eye, 8 * eye], 0).to(torch.bfloat16)[None, None].repeat(B, H, 1, 1).to(dev)
    o, lse = fa.attention_fwd(q, k, v, 1.0, False, p_drop=p, seed=seed)
    dvs = []
    for m in range(2):
        do = torch.zeros(N, d)
        do[64 * m:64 * m + 64] = eye
        do = do.to(torch.bfloat16)[None, None].repeat(B, H, 1, 1).to(dev)
        dvs.append(fa.attention_bwd(q, k, v, o, do, lse, 1.0, False, p_drop=p, seed=seed)[2])
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    t, s = oracle.threshold(p)
    unit = s / N
    for h in range(H):
        keep, _ = oracle.keep_mask(seed, h, N, p)
        keep = keep.astype(np.int64)
        code = np.rint(o[0, h].float().cpu().numpy() / unit).astype(np.int64)     # [N, 64]
        want = keep[:, :64] + 2 * keep[:, 64:128] + 4 * keep[:, 128:192] + 8 * keep[:, 192:]
        assert np.array_equal(code, want), f"forward mask differs for head {h}"
        for m in range(2):
            got_t = np.rint(dvs[m][0, h].float().cpu().numpy() / unit).astype(np.int64)   # [keys, 64 queries]
            assert np.array_equal(got_t, keep[64 * m:64 * m + 64, :].T), f"backward mask differs for head {h}, queries {64 * m}+"


def test_dropout_probability_validated(fa):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=dev)
    for bad in (-0.1, 1.0, float("nan"), 0.999):
        with pytest.raises(fa.FlashAttnError):
            fa.attention_fwd(q, q, q, 0.1, p_drop=bad, seed=1)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
