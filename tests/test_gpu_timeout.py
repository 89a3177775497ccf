"""The timeout path of the kernels' bounded waits, run for real.

Every wait of a kernel on an on-chip barrier gives up after a limit, records
FA_ERR_DEVICE_TIMEOUT in the device error word, and the kernel then lets the
copies and tensor-core operations it has issued finish, frees its tensor
memory and exits, instead of hanging. fa_options.test_stall = 1 makes the
kernels' tile loader stop after its first tile, so that a consumer's wait
runs out (after a short fa_options.wait_limit_us); nothing faults. The test
checks the reported status and site, and that the next normal call on the
same device gives the bits of a fresh run (a CTA that kept its tensor memory
would make that call's allocation wait forever; a wrong drain would corrupt
it).
"""
import math

import pytest
import torch

from exact_io_aware_39_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

FA_ERR_DEVICE_TIMEOUT = 5
LIMIT_US = 20000   # 20 ms per wait


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_39_gb300 as pkg
    from exact_io_aware_39_gb300 import build as b
    pkg.load(b.build())
    return pkg


def _inputs(d, causal):
    w = Workload("stall", 2, 3, 640, d, causal, 1.0 / math.sqrt(d))
    c = make_case(w, seed=11)
    dev = torch.device("cuda:0")
    return w, [c[n].to(dev) for n in ("q", "k", "v", "do")]


def _bits(t):
    return t.view(torch.int16) if t.dtype in (torch.bfloat16, torch.float16) else t.view(torch.int32)


@pytest.mark.parametrize("d,causal", [(64, True), (128, False), (256, True)])
def test_forward_wait_runs_out_and_device_stays_usable(fa, d, causal):
    w, (q, k, v, _) = _inputs(d, causal)
    assert fa.device_error()[0] == 0
    o0, l0 = fa.attention_fwd(q, k, v, w.scale, causal)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    fa.attention_fwd(q, k, v, w.scale, causal, wait_limit_us=LIMIT_US, test_stall=1)
    torch.cuda.synchronize()
    st, detail = fa.device_error()
    assert st == FA_ERR_DEVICE_TIMEOUT, detail
    assert detail[0] == FA_ERR_DEVICE_TIMEOUT and detail[1] < 100, detail   # a forward-kernel site
    assert fa.device_error()[0] == 0                                        # reading clears the word
    o1, l1 = fa.attention_fwd(q, k, v, w.scale, causal)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    assert torch.equal(_bits(o1), _bits(o0)) and torch.equal(_bits(l1), _bits(l0))


@pytest.mark.parametrize("d,causal", [(64, True), (128, False), (256, True)])
def test_backward_wait_runs_out_and_device_stays_usable(fa, d, causal):
    w, (q, k, v, do) = _inputs(d, causal)
    o, lse = fa.attention_fwd(q, k, v, w.scale, causal)
    dq0, dk0, dv0 = fa.attention_bwd(q, k, v, o, do, lse, w.scale, causal)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    fa.attention_bwd(q, k, v, o, do, lse, w.scale, causal, wait_limit_us=LIMIT_US, test_stall=1)
    torch.cuda.synchronize()
    st, detail = fa.device_error()
    assert st == FA_ERR_DEVICE_TIMEOUT, detail
    assert detail[0] == FA_ERR_DEVICE_TIMEOUT and 100 <= detail[1] < 200, detail   # a backward-kernel site
    dq1, dk1, dv1 = fa.attention_bwd(q, k, v, o, do, lse, w.scale, causal)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    # dK and dV are computed whole by one CTA per key tile: the same bits;
    # dQ partials are added in arrival order: the same values within rounding
    assert torch.equal(_bits(dk1), _bits(dk0)) and torch.equal(_bits(dv1), _bits(dv0))
    assert torch.allclose(dq1.float(), dq0.float(), rtol=1e-2, atol=1e-3)


@pytest.mark.parametrize("d", [64, 128])
def test_dropout_kernels_wait_runs_out_and_device_stays_usable(fa, d):
    """The dropout instances run other warp layouts (the backward's four P/dS
    warpgroups, which at d = 64 agree across all sixteen compute warps): the
    same stalled loader ends both kernels with a timeout, and the next calls
    give the bits of a fresh run."""
    w, (q, k, v, do) = _inputs(d, True)
    kw = dict(p_drop=0.2, seed=77)
    o0, l0 = fa.attention_fwd(q, k, v, w.scale, True, **kw)
    dq0, dk0, dv0 = fa.attention_bwd(q, k, v, o0, do, l0, w.scale, True, **kw)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    fa.attention_fwd(q, k, v, w.scale, True, wait_limit_us=LIMIT_US, test_stall=1, **kw)
    torch.cuda.synchronize()
    st, detail = fa.device_error()
    assert st == FA_ERR_DEVICE_TIMEOUT and detail[1] < 100, detail
    fa.attention_bwd(q, k, v, o0, do, l0, w.scale, True, wait_limit_us=LIMIT_US, test_stall=1, **kw)
    torch.cuda.synchronize()
    st, detail = fa.device_error()
    assert st == FA_ERR_DEVICE_TIMEOUT and 100 <= detail[1] < 200, detail
    o1, l1 = fa.attention_fwd(q, k, v, w.scale, True, **kw)
    dq1, dk1, dv1 = fa.attention_bwd(q, k, v, o1, do, l1, w.scale, True, **kw)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    assert torch.equal(_bits(o1), _bits(o0)) and torch.equal(_bits(l1), _bits(l0))
    assert torch.equal(_bits(dk1), _bits(dk0)) and torch.equal(_bits(dv1), _bits(dv0))

