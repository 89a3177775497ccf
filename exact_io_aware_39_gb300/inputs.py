"""Seeded synthetic inputs for exact attention, shared by the oracle tests,
the GPU parity tests and the bench.

This module holds no attention arithmetic: it only draws random numbers and
names the workloads. The workloads borrow the shapes of the pages' experiments
(one GPT-2-medium attention layer, a BERT-large padded batch, Path-X's 16K
length, block-sparse FlashAttention) and replace their data with N(0,1) values,
because the experiments' datasets and trained weights are not part of the
method.

Recipe (fixed, so that every consumer sees the same bits):
  * Q, K, V, dO: one CPU ``torch.Generator`` seeded with ``seed`` (default 0),
    ``randn`` in float32 drawn in the order Q, K, V, dO, each of shape
    [B, H, N, d], then rounded to bfloat16 (round-to-nearest-even).
  * kv_len (padded batches): a second generator seeded with ``seed + 1``,
    ``randint(lo, hi + 1)`` -> int32 [B], uniform on the inclusive range.
  * block_mask (block-sparse): a third generator seeded with ``seed + 2``,
    ``bernoulli(p)`` over an nT x nT grid of 128 x 128 blocks, uint8, with the
    diagonal forced to 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import torch

TILE = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    scale: float
    kv_len_range: tuple | None = None     # inclusive (lo, hi) or None
    block_p: float | None = None          # Bernoulli p of the block mask or None
    note: str = field(default="", compare=False)


# The five workloads: shapes from the pages' experiments, data synthetic.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 256, 64, False, 1.0 / math.sqrt(64),
                     note="exact-attention check, no mask"),
    "gpt2m": Workload("gpt2m", 8, 16, 1024, 64, True, 1.0 / 8.0,
                      note="GPT-2-medium attention layer shape, causal"),
    "bert_pad": Workload("bert_pad", 32, 16, 512, 64, False, 1.0 / 8.0,
                         kv_len_range=(128, 512),
                         note="BERT-large-style padded batch, per-sequence key length"),
    "long_causal": Workload("long_causal", 1, 32, 16384, 128, True, 1.0 / math.sqrt(128),
                            note="long-context causal, Path-X length"),
    "block_sparse": Workload("block_sparse", 4, 16, 4096, 64, False, 1.0 / 8.0,
                             block_p=0.25,
                             note="128x128 block mask, diagonal on, others Bernoulli(0.25)"),
}
WORKLOAD_ORDER = ["tiny", "gpt2m", "bert_pad", "long_causal", "block_sparse"]


def n_tiles(N: int) -> int:
    return (N + TILE - 1) // TILE


def draw_qkvdo(B, H, N, d, seed=0, dtype=torch.bfloat16):
    """Q, K, V, dO as 16-bit CPU tensors [B, H, N, d] (bfloat16 unless dtype
    says otherwise), drawn in that order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = []
    for _ in range(4):
        t = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        out.append(t.to(dtype))
    return tuple(out)


def draw_kv_len(B, lo, hi, seed=1):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def draw_block_mask(N, p, seed=2):
    nT = n_tiles(N)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    m = torch.bernoulli(torch.full((nT, nT), float(p)), generator=g).to(torch.uint8)
    idx = torch.arange(nT)
    m[idx, idx] = 1
    return m


def make_case(w: Workload, seed=0, B=None, H=None, N=None, dtype=torch.bfloat16):
    """All inputs of one workload (optionally with B, H or N overridden).

    Returns a dict of CPU tensors: q, k, v, do (bf16), kv_len (int32 [B] or
    None), block_mask (uint8 [nT, nT] or None), plus the scalar parameters.
    """
    B = w.B if B is None else B
    H = w.H if H is None else H
    N = w.N if N is None else N
    q, k, v, do = draw_qkvdo(B, H, N, w.d, seed, dtype)
    kv_len = None
    if w.kv_len_range is not None:
        lo, hi = w.kv_len_range
        kv_len = draw_kv_len(B, min(lo, N), min(hi, N), seed + 1)
    block_mask = None
    if w.block_p is not None:
        block_mask = draw_block_mask(N, w.block_p, seed + 2)
    return dict(q=q, k=k, v=v, do=do, kv_len=kv_len, block_mask=block_mask,
                B=B, H=H, N=N, d=w.d, scale=w.scale, causal=w.causal)
