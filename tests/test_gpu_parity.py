"""GPU parity: the CUDA path through the C ABI against the CPU float64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs):
  O    max-abs error        <= 1e-2
  LSE  max-abs error        <= 1e-3
  dQ, dK, dV  relative Frobenius error <= 2e-2
  tile states               bit-exact
Small shapes span several tiles and ragged tails; the five workloads run in
the launch configuration the bench times, compared in full where the oracle
finishes in seconds and on sampled heads otherwise.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_39_gb300.inputs import WORKLOADS, WORKLOAD_ORDER, Workload, make_case

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


def _run_gpu(fa, c, with_bwd=True):
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
    bm = None if c["block_mask"] is None else c["block_mask"].to(dev)
    # NaN canaries: every output element must be written
    o = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    fa.attention_fwd(q, k, v, c["scale"], c["causal"], kv, bm, out=o, lse=lse)
    res = dict(O=o, LSE=lse)
    if with_bwd:
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        need = fa.flash_attn_bwd_workspace_size(*q.shape)
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)   # garbage workspace
        fa.attention_bwd(q, k, v, o, do, lse, c["scale"], c["causal"], kv, bm, workspace=ws,
                         dq=dq, dk=dk, dv=dv)
        res.update(dQ=dq, dK=dk, dV=dv)
    torch.cuda.synchronize()
    st, detail = fa.device_error()
    assert st == 0, f"device error word {detail}"
    return {n: t.float().cpu().numpy() for n, t in res.items()}


def _compare(got, ref, heads=None, with_bwd=True, o_tol=O_TOL, o_rel=0.0):
    """o_rel > 0 adds o_rel * |O_ref| to the O bound element by element (the
    bf16 rounding of O itself, for cases whose rows can reach |O| > 2.5)."""
    B, H = ref["O"].shape[:2]
    sel = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    bi = np.array([b for b, _ in sel])
    hi = np.array([h for _, h in sel])
    for name in ("O", "LSE") + (("dQ", "dK", "dV") if with_bwd else ()):
        assert np.isfinite(got[name]).all() or name == "LSE", f"{name} has non-finite values"
    o_diff = np.abs(got["O"][bi, hi] - ref["O"][bi, hi])
    o_err = (o_diff - o_rel * np.abs(ref["O"][bi, hi])).max()
    r_lse, g_lse = ref["LSE"][bi, hi], got["LSE"][bi, hi]
    assert np.array_equal(np.isneginf(r_lse), np.isneginf(g_lse)), "fully masked rows differ"
    fin = np.isfinite(r_lse)
    lse_err = np.abs(g_lse[fin] - r_lse[fin]).max() if fin.any() else 0.0
    errs = dict(O=o_err, LSE=lse_err)
    if with_bwd:
        for name in ("dQ", "dK", "dV"):
            r, g = ref[name][bi, hi], got[name][bi, hi]
            nr = np.linalg.norm(r)
            errs[name] = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    # measured errors next to their bounds (visible with pytest -s), so that
    # the slack of every case is on record
    o_bound = f"{o_tol:g}" + (f" + {o_rel:.3g}|O_ref|" if o_rel else "")
    print(f"PARITY O {o_diff.max():.3e} (excess over the |O_ref| term {o_err:.3e}, bound {o_bound}) "
          f"LSE {lse_err:.3e} (bound {LSE_TOL:g})"
          + "".join(f" {n} {errs[n]:.3e}" for n in ("dQ", "dK", "dV") if n in errs)
          + (f" (bound {GRAD_TOL:g})" if with_bwd else ""))
    assert o_err <= o_tol, errs
    assert lse_err <= LSE_TOL, errs
    if with_bwd:
        for name in ("dQ", "dK", "dV"):
            assert errs[name] <= GRAD_TOL, errs
    return errs


SMALL = [
    # name, B, H, N, d, causal, kv_len, block mask (None / "rand")
    ("single_tile", 1, 1, 128, 64, False, None, None),
    ("tiny_noncausal", 1, 2, 256, 64, False, None, None),
    ("ragged_tail", 2, 3, 300, 64, False, None, None),
    ("ragged_causal", 2, 2, 333, 64, True, None, None),
    ("d128", 1, 2, 384, 128, False, None, None),
    ("d128_causal_ragged", 1, 3, 520, 128, True, None, None),
    ("odd_tiles_causal", 1, 2, 640, 64, True, None, None),
    ("n1", 2, 2, 1, 64, False, None, None),
    ("n129_causal", 1, 2, 129, 128, True, None, None),
    ("kv_len_mixed", 4, 2, 384, 64, False, [1, 384, 200, 129], None),
    ("kv_len_zero_rows", 3, 2, 256, 64, False, [0, 77, 256], None),
    ("kv_len_causal_d128", 3, 2, 300, 128, True, [300, 5, 130], None),
    ("block_mask", 2, 2, 768, 64, False, None, "rand"),
    ("block_mask_causal_d128", 1, 2, 640, 128, True, None, "rand"),
    ("block_mask_empty_rows", 1, 2, 512, 64, False, None, "rows"),
    ("all_masks", 2, 2, 700, 64, True, [650, 300], "rand"),
]


def _small_case(name, B, H, N, d, causal, kv, bm, dtype=torch.bfloat16):
    w = Workload(name, B, H, N, d, causal, 1.0 / math.sqrt(d))
    c = make_case(w, seed=zlib.crc32(name.encode()) % 1000, dtype=dtype)
    if kv is not None:
        c["kv_len"] = torch.tensor(kv, dtype=torch.int32)
    nT = (N + 127) // 128
    if bm == "rand":
        g = torch.Generator().manual_seed(5)
        m = (torch.rand(nT, nT, generator=g) < 0.5).to(torch.uint8)
        m[torch.arange(nT), torch.arange(nT)] = 1
        c["block_mask"] = m
    elif bm == "rows":   # query tile 1 has no live block at all
        m = torch.ones(nT, nT, dtype=torch.uint8)
        m[1, :] = 0
        m[0, 2] = 0
        c["block_mask"] = m
    return c


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_small_shapes_match_oracle(fa, spec):
    c = _small_case(*spec)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"],
                                   c["kv_len"], c["block_mask"])
    _compare(got, ref)


# The backward kernel is persistent (one CTA per SM, each walking several
# (key tile, batch-head) items with its pipeline running on across them):
# shapes with more than twice as many key-tile items as SMs, including items
# whose key tile has no live query tile (kv_len 0 and short lengths) and
# block-sparse rows, compared in full.
MANY_ITEMS = [
    # name, B, N, d, causal, kv_len, block mask; H is chosen so that B * H * nT > 2.2 x SMs
    ("many_items_kv_len_causal", 4, 512, 64, True, [512, 0, 300, 129], None),
    ("many_items_d128_kv_len", 2, 384, 128, False, [384, 200], None),
    ("many_items_block_mask", 2, 512, 64, False, None, "rand"),
    ("many_items_d96_all_masks", 2, 640, 96, True, [600, 333], "rand"),
    ("many_items_d256_kv_len_causal", 4, 512, 256, True, [512, 0, 300, 129], None),
    ("many_items_d192_block_mask", 2, 512, 192, False, None, "rand"),
]


@pytest.mark.parametrize("spec", MANY_ITEMS, ids=[s[0] for s in MANY_ITEMS])
def test_many_items_per_cta_match_oracle(fa, spec):
    name, B, N, d, causal, kv, bm = spec
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nT = (N + 127) // 128
    H = max(2, math.ceil(2.2 * sms / (B * nT)))
    assert B * H * nT > 2 * sms
    c = _small_case(name, B, H, N, d, causal, kv, bm)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"],
                                   c["kv_len"], c["block_mask"])
    _compare(got, ref, o_rel=HEAD_DIM_O_REL if d not in (64, 128) else 0.0)


# O bound of the head-dimension cases: 1e-2 plus the bf16 rounding of O itself
# (8 significant bits: up to 2^-8 |O|), since rows that see only a few keys
# (kv_len = 5) reach |O| > 2.5, where rounding alone approaches 1e-2.
HEAD_DIM_O_REL = 2.0 ** -8

HEAD_DIMS = [
    # head dimensions other than 64 and 128 run on the 64- or 128-column
    # kernels over zero-padded columns
    ("d8", 1, 2, 256, 8, False, None, None),
    ("d32_causal_ragged", 2, 2, 333, 32, True, None, None),
    ("d40_kv_len", 3, 2, 300, 40, False, [300, 5, 130], None),
    ("d72", 1, 2, 384, 72, False, None, None),
    ("d96_causal_block_mask", 1, 2, 640, 96, True, None, "rand"),
    ("d120_all_masks", 2, 2, 700, 120, True, [650, 300], "rand"),
    # above 128: the wide kernels (one Q tile per forward CTA; the backward
    # split over the two halves of the head dimension)
    ("d136_causal_ragged", 1, 2, 333, 136, True, None, None),
    ("d160_causal", 1, 2, 640, 160, True, None, None),
    ("d160_kv_len", 3, 2, 300, 160, False, [300, 5, 130], None),
    ("d192_block_mask", 2, 2, 768, 192, False, None, "rand"),
    ("d192_causal_block_mask", 1, 2, 640, 192, True, None, "rand"),
    ("d256", 1, 2, 384, 256, False, None, None),
    ("d256_causal_kv_len", 3, 2, 520, 256, True, [520, 77, 300], None),
    ("d256_block_mask_empty_rows", 1, 2, 512, 256, False, None, "rows"),
    ("d248_all_masks", 2, 2, 700, 248, True, [650, 300], "rand"),
    ("d256_n1", 2, 2, 1, 256, False, None, None),
]


@pytest.mark.parametrize("spec", HEAD_DIMS, ids=[s[0] for s in HEAD_DIMS])
def test_head_dims_match_oracle(fa, spec):
    c = _small_case(*spec)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"],
                                   c["kv_len"], c["block_mask"])
    _compare(got, ref, o_rel=HEAD_DIM_O_REL)


@pytest.mark.parametrize("d", [96, 256])
def test_head_dim_fp16(fa, d):
    c = _small_case(f"d{d}_fp16", 1, 2, 384, d, True, None, None, dtype=torch.float16)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"])
    _compare(got, ref, o_rel=HEAD_DIM_O_REL)


@pytest.mark.parametrize("spec", [h for h in HEAD_DIMS if h[4] > 128], ids=[h[0] for h in HEAD_DIMS if h[4] > 128])
def test_wide_kernels_compute_exactly_the_classified_tiles(fa, spec):
    """The tile record of the wide kernels (d > 128) against the oracle's
    tile states, as for the narrower kernels."""
    c = _small_case(*spec)
    rec_f, rec_b = _recorded_tiles(fa, c)
    want = oracle.tile_states(c["B"], c["N"], c["causal"], c["kv_len"], c["block_mask"])
    want = np.broadcast_to(want[:, None], rec_f.shape)
    assert np.array_equal(rec_f, want)
    assert np.array_equal(rec_b, want)


def test_wide_head_dims_refuse_dropout(fa):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 128, 256, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FlashAttnError):
        fa.attention_fwd(q, q, q, 0.1, p_drop=0.1)
    assert fa.device_error()[0] == 0


MAX_LEN = [
    # the longest supported sequence (131072 keys), and a ragged length just below it
    (131072, 64),
    (131071, 128),
]


@pytest.mark.parametrize("N,d", MAX_LEN, ids=[f"N{n}_d{d}" for n, d in MAX_LEN])
def test_maximum_length_sampled_rows(fa, N, d):
    """Causal attention at the maximum length, compared on sampled query rows
    (O, LSE, dQ) and on key rows near the end (dK, dV: under the causal mask
    they need only the rows after them), computed by the oracle row block by
    row block. O bound as for the head-dimension cases (early causal rows
    average two or three values, |O| > 2.5)."""
    c = _small_case(f"maxlen_{N}_{d}", 1, 1, N, d, True, None, None)
    got = _run_gpu(fa, c)
    rows = [0, 1, 127, 128, 4097, N // 2, N - 129, N - 1]
    keys = [N - 1, N - 2, N - 130, N - 300]
    ref = oracle.head_rows(c["q"][0, 0], c["k"][0, 0], c["v"][0, 0], c["do"][0, 0], c["scale"], True,
                           rows, keys)
    o_ref = ref["O"]
    o_got = got["O"][0, 0][rows]
    assert (np.abs(o_got - o_ref) - HEAD_DIM_O_REL * np.abs(o_ref)).max() <= O_TOL
    assert np.abs(got["LSE"][0, 0][rows] - ref["LSE"]).max() <= LSE_TOL
    for name, idx in (("dQ", rows), ("dK", keys), ("dV", keys)):
        g, r = got[name][0, 0][idx], ref[name]
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert rel <= GRAD_TOL, (name, rel)


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_tile_map_bit_exact(fa, spec):
    c = _small_case(*spec)
    dev = torch.device("cuda:0")
    kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
    bm = None if c["block_mask"] is None else c["block_mask"].to(dev)
    got = fa.tile_map(c["B"], c["N"], c["causal"], kv, bm).cpu().numpy()
    want = oracle.tile_states(c["B"], c["N"], c["causal"], c["kv_len"], c["block_mask"])
    assert np.array_equal(got, want)


def _recorded_tiles(fa, c, p_drop=0.0):
    """The tiles the forward and the backward kernels computed, as recorded
    through fa_options.tile_record: two uint8 arrays [B, H, nT, nT]."""
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
    bm = None if c["block_mask"] is None else c["block_mask"].to(dev)
    B, H, N = q.shape[:3]
    nT = (N + 127) // 128
    rec_f = torch.zeros((B, H, nT, nT), dtype=torch.uint8, device=dev)
    rec_b = torch.zeros_like(rec_f)
    kw = dict(p_drop=p_drop, seed=5) if p_drop > 0 else {}
    o, lse = fa.attention_fwd(q, k, v, c["scale"], c["causal"], kv, bm, tile_record=rec_f, **kw)
    fa.attention_bwd(q, k, v, o, do, lse, c["scale"], c["causal"], kv, bm, tile_record=rec_b, **kw)
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    return rec_f.cpu().numpy(), rec_b.cpu().numpy()


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_kernels_compute_exactly_the_classified_tiles(fa, spec):
    """The tile-skip set as the kernels ran it: every (b, h, qi, kj) the
    forward and the backward kernel computed, recorded by the thread that
    decides on element masking (1 unmasked, 2 masked, summed over visits),
    equals the oracle's tile states for every head, bit for bit; a skipped
    tile that was computed, a masked tile computed without masking, or a tile
    computed twice would all differ."""
    c = _small_case(*spec)
    rec_f, rec_b = _recorded_tiles(fa, c)
    want = oracle.tile_states(c["B"], c["N"], c["causal"], c["kv_len"], c["block_mask"])
    want = np.broadcast_to(want[:, None], rec_f.shape)
    assert np.array_equal(rec_f, want)
    assert np.array_equal(rec_b, want)


@pytest.mark.parametrize("spec", [s for s in SMALL if s[4] <= 128], ids=[s[0] for s in SMALL if s[4] <= 128])
def test_dropout_kernels_compute_exactly_the_classified_tiles(fa, spec):
    """The same record from the dropout instances (other warp layouts in the
    backward: four P/dS warpgroups)."""
    c = _small_case(*spec)
    rec_f, rec_b = _recorded_tiles(fa, c, p_drop=0.2)
    want = oracle.tile_states(c["B"], c["N"], c["causal"], c["kv_len"], c["block_mask"])
    want = np.broadcast_to(want[:, None], rec_f.shape)
    assert np.array_equal(rec_f, want)
    assert np.array_equal(rec_b, want)


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workload_kernels_compute_exactly_the_classified_tiles(fa, name):
    """The same record on the five workloads in their bench launch
    configuration (heads reduced where the record would not change: the
    states are shared by all heads; long_causal keeps its 128 x 128 grid)."""
    w = WORKLOADS[name]
    c = make_case(w, H=min(w.H, 2))
    rec_f, rec_b = _recorded_tiles(fa, c)
    want = oracle.tile_states(c["B"], w.N, w.causal, c["kv_len"], c["block_mask"])
    want = np.broadcast_to(want[:, None], rec_f.shape)
    assert np.array_equal(rec_f, want)
    assert np.array_equal(rec_b, want)


def test_plain_signatures_match_oracle(fa):
    """flash_attn_fwd and flash_attn_bwd themselves (the calls without
    options), through ctypes with raw device pointers, on a case with every
    mask kind and a ragged tail."""
    c = _small_case("plain_abi", 2, 2, 700, 64, True, [650, 300], "rand")
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kv, bm = c["kv_len"].to(dev), c["block_mask"].to(dev)
    B, H, N, d = q.shape
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    need = fa.flash_attn_bwd_workspace_size(B, H, N, d)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)
    P = fa._lib._ptr
    s = fa._lib._stream(None)
    st = fa.flash_attn_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, c["scale"], 1, P(kv), P(bm), s)
    assert st == 0
    st = fa.flash_attn_bwd(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), B, H, N, d, c["scale"], 1,
                           P(kv), P(bm), P(ws), need, s)
    assert st == 0
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    got = {n: t.float().cpu().numpy() for n, t in dict(O=o, LSE=lse, dQ=dq, dK=dk, dV=dv).items()}
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], True, c["kv_len"],
                                   c["block_mask"])
    _compare(got, ref)


FP16 = [s for s in SMALL if s[0] in ("tiny_noncausal", "ragged_causal", "d128_causal_ragged",
                                      "kv_len_mixed", "block_mask_causal_d128", "all_masks")]


@pytest.mark.parametrize("spec", FP16, ids=[s[0] for s in FP16])
def test_fp16_matches_oracle(fa, spec):
    """The fp16 element type (fa_options.dtype = FA_DTYPE_F16): same kernels,
    same tolerances."""
    c = _small_case(*spec, dtype=torch.float16)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], c["scale"], c["causal"],
                                   c["kv_len"], c["block_mask"])
    _compare(got, ref)


def test_fp16_long_causal_sampled_heads(fa):
    w = WORKLOADS["long_causal"]
    c = make_case(w, dtype=torch.float16)
    got = _run_gpu(fa, c)
    heads = [(0, 5), (0, 20)]
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], w.scale, w.causal, heads=heads)
    _compare(got, ref, heads=heads)


# heads compared per workload: all where the oracle is quick, else a sample
HEADS = {
    "tiny": None,
    "gpt2m": None,
    "bert_pad": None,
    "long_causal": [(0, 0), (0, 31)],
    "block_sparse": [(0, 0), (1, 7), (2, 11), (3, 15)],
}


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workloads_match_oracle(fa, name):
    w = WORKLOADS[name]
    c = make_case(w)
    got = _run_gpu(fa, c)
    ref = oracle.attention_fwd_bwd(c["q"], c["k"], c["v"], c["do"], w.scale, w.causal,
                                   c["kv_len"], c["block_mask"], heads=HEADS[name])
    errs = _compare(got, ref, heads=HEADS[name])
    print(name, {k: float(v) for k, v in errs.items()})


@pytest.mark.parametrize("name", WORKLOAD_ORDER)
def test_workload_tile_map_bit_exact(fa, name):
    w = WORKLOADS[name]
    c = make_case(w, H=1)
    dev = torch.device("cuda:0")
    kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
    bm = None if c["block_mask"] is None else c["block_mask"].to(dev)
    got = fa.tile_map(c["B"], w.N, w.causal, kv, bm).cpu().numpy()
    want = oracle.tile_states(c["B"], w.N, w.causal, c["kv_len"], c["block_mask"])
    assert np.array_equal(got, want)


def test_repeat_calls_are_deterministic_and_leave_guards(fa):
    """Same inputs twice give the same bits for O, LSE, dK and dV (dQ is
    summed with atomic adds, so only its values within rounding repeat);
    bytes around every output stay untouched (outputs are views into larger
    guarded buffers)."""
    c = _small_case("guards", 2, 2, 300, 128, True, [300, 150], None)
    dev = torch.device("cuda:0")
    q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
    kv = c["kv_len"].to(dev)
    n = q.numel()
    G = 4096

    def guarded(numel, dtype):
        buf = torch.full((numel + 2 * G,), 7, dtype=dtype, device=dev)
        return buf, buf[G:G + numel]

    outs = []
    for _ in range(2):
        ob, o = guarded(n, torch.bfloat16)
        lb, l = guarded(n // q.shape[-1], torch.float32)
        gb = [guarded(n, torch.bfloat16) for _ in range(3)]
        fa.attention_fwd(q, k, v, c["scale"], True, kv, None, out=o.view_as(q), lse=l.view(q.shape[:3]))
        fa.attention_bwd(q, k, v, o.view_as(q), do, l.view(q.shape[:3]), c["scale"], True, kv, None,
                         dq=gb[0][1].view_as(q), dk=gb[1][1].view_as(q), dv=gb[2][1].view_as(q))
        torch.cuda.synchronize()
        for buf in [ob, lb] + [x[0] for x in gb]:
            assert (buf[:G] == 7).all() and (buf[-G:] == 7).all()
        outs.append([o.clone(), l.clone()] + [x[1].clone() for x in gb])
    for idx, (a, b) in enumerate(zip(*outs)):
        if idx == 2:   # dQ
            assert torch.allclose(a.float(), b.float(), rtol=1e-2, atol=1e-3)
        else:
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
    assert fa.device_error()[0] == 0


def test_concurrent_backward_calls_on_two_streams(fa):
    """The persistent backward kernel hands out its work items from a counter
    in the caller's workspace: two calls in flight at once on two streams,
    each with its own workspace, give the bits of the same calls run one
    after the other for dK and dV (each item is computed whole by one CTA)
    and dQ within rounding (partials are added in arrival order)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = max(2, math.ceil(2.2 * sms / (2 * 4)))
    cases = [_small_case("streams_a", 2, H, 512, 64, True, None, None),
             _small_case("streams_b", 2, H, 512, 128, False, [512, 260], None)]
    dev = torch.device("cuda:0")
    prepared = []
    for c in cases:
        q, k, v, do = (c[n].to(dev) for n in ("q", "k", "v", "do"))
        kv = None if c["kv_len"] is None else c["kv_len"].to(dev)
        o, lse = fa.attention_fwd(q, k, v, c["scale"], c["causal"], kv, None)
        prepared.append((c, q, k, v, do, kv, o, lse))

    def run(args, stream, ws):
        c, q, k, v, do, kv, o, lse = args
        return fa.attention_bwd(q, k, v, o, do, lse, c["scale"], c["causal"], kv, None, workspace=ws,
                                stream=stream)

    workspaces = [torch.empty(fa.flash_attn_bwd_workspace_size(*a[1].shape), dtype=torch.uint8, device=dev)
                  for a in prepared]
    serial = [run(a, torch.cuda.current_stream(), ws) for a, ws in zip(prepared, workspaces)]
    torch.cuda.synchronize()
    serial = [[t.clone() for t in r] for r in serial]
    streams = [torch.cuda.Stream(device=dev) for _ in prepared]
    for s_ in streams:
        s_.wait_stream(torch.cuda.current_stream())
    together = []
    for _ in range(3):
        for a, ws, s_ in zip(prepared, workspaces, streams):
            with torch.cuda.stream(s_):
                together.append(run(a, s_, ws))
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
    for rep in range(3):
        for i in range(len(prepared)):
            dq, dk, dv = together[2 * rep + i]
            assert torch.equal(dk.view(torch.int16), serial[i][1].view(torch.int16))
            assert torch.equal(dv.view(torch.int16), serial[i][2].view(torch.int16))
            assert torch.allclose(dq.float(), serial[i][0].float(), rtol=1e-2, atol=1e-3)


def test_invalid_arguments_on_device(fa):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 128, dtype=torch.float32, device=dev)
    P = fa._lib._ptr
    s = fa._lib._stream(None)
    for bad_d in (60, 264):   # rejected before anything is launched
        assert fa.flash_attn_fwd(P(q), P(q), P(q), P(q), P(lse), 1, 1, 128, bad_d, 0.1, 0, None, None, s) == 2
    mis = torch.zeros(1 + 128 * 64, dtype=torch.bfloat16, device=dev)[1:]
    assert fa.flash_attn_fwd(P(mis), P(q), P(q), P(q), P(lse), 1, 1, 128, 64, 0.1, 0, None, None, s) == 1
    need = fa.flash_attn_bwd_workspace_size(1, 1, 128, 64)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    args = [P(q)] * 5 + [P(lse)] + [P(q)] * 3 + [1, 1, 128, 64, 0.1, 0, None, None]
    assert fa.flash_attn_bwd(*args, P(ws), need - 16, s) == 3
    torch.cuda.synchronize()
    assert fa.device_error()[0] == 0
