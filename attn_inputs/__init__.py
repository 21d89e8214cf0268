"""Seeded synthetic inputs for the attention forward pass.

This module only draws random numbers and packs them into the layouts the
attention calls take. It holds none of the attention arithmetic, so both the
CPU oracle and the CUDA path can be fed from it without sharing any of the
method's code.

Layouts
-------
* fixed length: ``q [B, N, H, d]``, ``k, v [B, N, Hkv, d]`` (BSHD, contiguous)
* packed variable length: ``q [T, H, d]``, ``k, v [T, Hkv, d]`` (THD) plus
  ``cu_seqlens`` (int32, ``nseq + 1`` prefix offsets, ``cu_seqlens[0] = 0``).

Distributions
-------------
* ``normal``: i.i.d. N(0, 1) drawn in fp32 and rounded to the storage dtype.
* ``outlier``: N(0, 1) plus, independently per entry with probability 0.001,
  an extra N(0, 100) term (variance 100, i.e. standard deviation 10). This is
  the heavy-tailed input used to study FP8 error with and without the
  incoherent-processing rotation.

Draw order is fixed: Q, then K, then V, each in row-major order, from one
``torch.Generator`` seeded with ``seed``.
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "DTYPES",
    "draw",
    "qkv_fixed",
    "qkv_varlen",
    "varlen_lengths",
    "cu_seqlens_from_lengths",
    "sample_rows",
]

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}

OUTLIER_PROB = 1e-3
OUTLIER_STD = 10.0


def draw(shape, gen: torch.Generator, dist: str = "normal") -> torch.Tensor:
    """One fp32 tensor of ``shape`` from ``gen`` with the named distribution."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "normal":
        return x
    if dist == "outlier":
        hit = torch.rand(shape, generator=gen, dtype=torch.float32) < OUTLIER_PROB
        extra = torch.randn(shape, generator=gen, dtype=torch.float32) * OUTLIER_STD
        return x + torch.where(hit, extra, torch.zeros_like(extra))
    raise ValueError(f"unknown distribution {dist!r}")


def qkv_fixed(B: int, N: int, H: int, Hkv: int, d: int, seed: int = 0,
              dtype: str = "bf16", dist: str = "normal"):
    """Q [B,N,H,d], K and V [B,N,Hkv,d] on the host in ``dtype``."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    t = DTYPES[dtype]
    q = draw((B, N, H, d), gen, dist).to(t)
    k = draw((B, N, Hkv, d), gen, dist).to(t)
    v = draw((B, N, Hkv, d), gen, dist).to(t)
    return q, k, v


def varlen_lengths(nseq: int = 8, lo: int = 1024, hi: int = 32768, seed: int = 0) -> np.ndarray:
    """Sequence lengths uniform on the integers [lo, hi] (both ends included)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, endpoint=True, size=nseq).astype(np.int64)


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=cu[1:])
    return cu.astype(np.int32)


def qkv_varlen(lengths, H: int, Hkv: int, d: int, seed: int = 0,
               dtype: str = "bf16", dist: str = "normal"):
    """Packed Q [T,H,d], K and V [T,Hkv,d] plus int32 ``cu_seqlens``."""
    cu = cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    gen = torch.Generator(device="cpu").manual_seed(seed)
    t = DTYPES[dtype]
    q = draw((T, H, d), gen, dist).to(t)
    k = draw((T, Hkv, d), gen, dist).to(t)
    v = draw((T, Hkv, d), gen, dist).to(t)
    return q, k, v, cu


def sample_rows(lengths, H: int, count: int, seed: int = 0):
    """A seeded sample of (sequence, head, row) triples for row-sampled checks.

    It always includes, for every sequence, rows 0, 127, 128 and the last row
    (where they exist) on a seeded head, and fills the rest uniformly.
    Returns three int64 arrays (seq, head, row), sorted and de-duplicated.
    """
    rng = np.random.default_rng(seed + 7919)
    lengths = np.asarray(lengths, dtype=np.int64)
    seqs, heads, rows = [], [], []
    for s, n in enumerate(lengths):
        for r in (0, 127, 128, int(n) - 1):
            if 0 <= r < n:
                seqs.append(s)
                heads.append(int(rng.integers(0, H)))
                rows.append(r)
    rest = max(0, count - len(rows))
    if rest:
        weights = lengths / lengths.sum()
        s_pick = rng.choice(len(lengths), size=rest, p=weights)
        seqs.extend(s_pick.tolist())
        heads.extend(rng.integers(0, H, size=rest).tolist())
        rows.extend([int(rng.integers(0, lengths[s])) for s in s_pick])
    trip = np.unique(np.stack([np.asarray(seqs), np.asarray(heads), np.asarray(rows)], axis=1), axis=0)
    return trip[:, 0].astype(np.int64), trip[:, 1].astype(np.int64), trip[:, 2].astype(np.int64)
