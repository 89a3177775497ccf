"""Numerical stability as the logits grow: the flash path against standard
attention with S and dP stored in fp32, and with S and dP stored in the 16-bit
input type (as a framework's 16-bit matmul returns them), all three against
the float64 oracle on the same bf16 inputs.

The pages say that with its online softmax and high-precision accumulators the
method is often numerically more stable than standard PyTorch attention
(FlashAttention proof-of-work page, the question whether the method is an
approximation). The flash path keeps S in fp32 on chip; a 16-bit S keeps 8
significant bits (bf16), so once |S| reaches tens, rounding S alone moves
exp(S - LSE) by whole percents. The logits are grown by multiplying Q by
alpha (Q stays bf16; the oracle sees the same rounded Q).

Checked: the flash path stays within its bounds at every alpha (O: 1e-2 +
2^-8 |O_ref| elementwise, the second term being the bf16 rounding of O; LSE
max-abs 1e-3; gradients 2e-2 relative Frobenius while alpha <= 4, where the
gradients are not dominated by near one-hot rows), and from alpha = 16 on its O
and LSE errors are below those of the 16-bit standard attention. Set
FA_STUDY_OUT to a file path to append the error table there.
"""
import math
import os
import zlib

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_39_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

ALPHAS = [1, 4, 16, 64]


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_io_aware_39_gb300 as pkg
    from exact_io_aware_39_gb300 import build as b
    pkg.load(b.build())
    return pkg


def _errors(got, ref):
    fin = np.isfinite(ref["LSE"])
    out = {"O": float(np.abs(got["O"] - ref["O"]).max()),
           "O_excess": float((np.abs(got["O"] - ref["O"]) - 2.0 ** -8 * np.abs(ref["O"])).max()),
           "LSE": float(np.abs(got["LSE"][fin] - ref["LSE"][fin]).max())}
    for n in ("dQ", "dK", "dV"):
        out[n] = float(np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n]))
    return out


@pytest.fixture(scope="module")
def table(fa):
    w = Workload("stability", 1, 2, 512, 64, False, 0.125)
    base = make_case(w, seed=zlib.crc32(b"stability") % 1000)
    dev = torch.device("cuda:0")
    rows = []
    for alpha in ALPHAS:
        q = (base["q"].float() * alpha).to(torch.bfloat16)
        k, v, do = base["k"], base["v"], base["do"]
        ref = oracle.attention_fwd_bwd(q, k, v, do, w.scale, False)
        gq, gk, gv, gdo = (t.to(dev) for t in (q, k, v, do))
        res = {}
        o, lse = fa.attention_fwd(gq, gk, gv, w.scale)
        dq, dk, dv = fa.attention_bwd(gq, gk, gv, o, gdo, lse, w.scale)
        res["flash"] = dict(O=o, LSE=lse, dQ=dq, dK=dk, dV=dv)
        for name, s16 in (("standard_fp32_S", False), ("standard_16bit_S", True)):
            o, lse, ws = fa.standard_attention_fwd(gq, gk, gv, w.scale, s16=s16)
            dq, dk, dv = fa.standard_attention_bwd(gq, gk, gv, gdo, ws, w.scale, s16=s16)
            res[name] = dict(O=o, LSE=lse, dQ=dq, dK=dk, dV=dv)
        torch.cuda.synchronize()
        assert fa.device_error()[0] == 0
        max_s = float(np.abs(np.einsum("bhid,bhjd->bhij", q.double().numpy(), k.double().numpy())).max() * w.scale)
        for name, r in res.items():
            got = {n: t.float().cpu().numpy() for n, t in r.items()}
            rows.append(dict(alpha=alpha, max_abs_S=max_s, path=name, **_errors(got, ref)))
    out = os.environ.get("FA_STUDY_OUT")
    if out:
        with open(out, "a") as f:
            f.write("| alpha | max abs S | path | O max-abs | LSE max-abs | dQ rel | dK rel | dV rel |\n")
            f.write("|---|---|---|---|---|---|---|---|\n")
            for r in rows:
                f.write(f"| {r['alpha']} | {r['max_abs_S']:.1f} | {r['path']} | {r['O']:.3e} | {r['LSE']:.3e} | "
                        f"{r['dQ']:.3e} | {r['dK']:.3e} | {r['dV']:.3e} |\n")
    return rows


def _row(table, alpha, path):
    return next(r for r in table if r["alpha"] == alpha and r["path"] == path)


@pytest.mark.parametrize("alpha", ALPHAS)
def test_flash_path_within_bounds(table, alpha):
    r = _row(table, alpha, "flash")
    assert r["O_excess"] <= 1e-2, r
    assert r["LSE"] <= 1e-3, r
    if alpha <= 4:
        assert max(r["dQ"], r["dK"], r["dV"]) <= 2e-2, r


@pytest.mark.parametrize("alpha", [a for a in ALPHAS if a >= 16])
def test_flash_more_accurate_than_16bit_standard(table, alpha):
    f = _row(table, alpha, "flash")
    s = _row(table, alpha, "standard_16bit_S")
    assert f["O"] < s["O"] and f["LSE"] < s["LSE"], (f, s)
