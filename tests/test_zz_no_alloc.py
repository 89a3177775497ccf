"""flash_attn_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (a plug-in inside another runtime's execute callback, a serving
loop that must not call cudaMalloc on the request path, a program whose
memory belongs to a pool with no raw buffers). It takes its scratch from a
fixed array inside the library instead of a caller-provided workspace.

Checked through the C ABI against flash_attn_bwd (which uses a workspace) on
the same inputs, twice in a row, since every call reuses the same array and
must not depend on what the previous call left in it; and after a call of a
larger shape, whose leftovers sit where the smaller call keeps its row
vectors and work counter. Both entry points run the same kernels in the same
launch sequence, so dK and dV agree bit for bit; dQ partials are added in
arrival order, so dQ agrees within rounding. Collected last, so a run that
stops at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from exact_io_aware_39_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

GRAD_TOL = 2e-2   # relative Frobenius error of dQ, as for the other gradient tests


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_39_gb300 as pkg
    from exact_io_aware_39_gb300 import build as b
    pkg.load(b.build())
    return pkg


def _rel(a, b):
    a, b = a.double(), b.double()
    nb = torch.linalg.norm(b)
    return float(torch.linalg.norm(a - b) / nb) if nb > 0 else float(torch.linalg.norm(a))


CASES = [
    # B, H, N, d, causal, kv_len, block mask
    (2, 4, 700, 64, True, [700, 333], False),
    (1, 3, 520, 128, False, None, True),
]


def _prepare(fa, case):
    B, H, N, d, causal, kv, use_bm = case
    w = Workload("noalloc", B, H, N, d, causal, 1.0 / math.sqrt(d))
    c = make_case(w, seed=3)
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kvt = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=dev)
    bm = None
    if use_bm:
        nT = (N + 127) // 128
        g = torch.Generator().manual_seed(9)
        m = (torch.rand(nT, nT, generator=g) < 0.5).to(torch.uint8)
        m[torch.arange(nT), torch.arange(nT)] = 1
        bm = m.to(dev)
    need = fa.flash_attn_bwd_workspace_size(B, H, N, d)
    assert 0 < need <= fa._lib.BWD_NOALLOC_SCRATCH_BYTES
    o, lse = fa.attention_fwd(q, k, v, w.scale, causal, kvt, bm)
    ref = fa.attention_bwd(q, k, v, o, do, lse, w.scale, causal, kvt, bm)
    return (q, k, v, o, do, lse, B, H, N, d, w.scale, causal, kvt, bm), ref


def _noalloc(fa, args):
    q, k, v, o, do, lse, B, H, N, d, scale, causal, kvt, bm = args
    P = fa._lib._ptr
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    st = fa.flash_attn_bwd_noalloc(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv),
                                   B, H, N, d, scale, int(causal), P(kvt), P(bm), fa._lib._stream(None))
    assert st == 0, fa.flash_attn_status_string(st)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    return dq, dk, dv


def _check_same(got, ref):
    dq, dk, dv = got
    for t in got:
        assert torch.isfinite(t.float()).all()
    assert torch.equal(dk.view(torch.int16), ref[1].view(torch.int16))
    assert torch.equal(dv.view(torch.int16), ref[2].view(torch.int16))
    assert _rel(dq.float(), ref[0].float()) <= GRAD_TOL


@pytest.mark.parametrize("case", CASES, ids=["d64_causal_kvlen", "d128_blockmask"])
def test_noalloc_matches_workspace_backward_twice(fa, case):
    args, ref = _prepare(fa, case)
    for _ in range(2):
        _check_same(_noalloc(fa, args), ref)


BIG = (2, 6, 900, 128, False, None, True)


def test_noalloc_after_a_larger_call(fa):
    """A larger call (d = 128, block mask, about four times the scratch of the
    d = 64 case) leaves its accumulator, row vectors and counter in the array;
    the smaller call that follows, whose sections start at other offsets, must
    not read any of it."""
    big, _ = _prepare(fa, BIG)
    small, ref_small = _prepare(fa, CASES[0])
    assert fa.flash_attn_bwd_workspace_size(*big[6:10]) > 2 * fa.flash_attn_bwd_workspace_size(*small[6:10])
    _noalloc(fa, big)
    _check_same(_noalloc(fa, small), ref_small)


def test_noalloc_rejects_shapes_beyond_its_scratch(fa):
    """A shape whose workspace exceeds the fixed scratch is refused before
    anything is launched (the pointers are never dereferenced)."""
    B, H, N, d = 1, 32, 16384, 128
    assert fa.flash_attn_bwd_workspace_size(B, H, N, d) > fa._lib.BWD_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(64, dtype=torch.float32, device="cuda:0")
    p = ctypes.c_void_p(t.data_ptr())
    st = fa.flash_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0.1, 1, None, None,
                                   fa._lib._stream(None))
    assert st == fa._lib.FA_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
