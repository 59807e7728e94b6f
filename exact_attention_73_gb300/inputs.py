"""Seeded synthetic inputs for exact attention.

This module holds random-number recipes only: it contains none of the
attention arithmetic, so both the float64 oracle (through the tests) and the
CUDA library (through the tests and the benchmark) may take their inputs from
it without sharing any part of the method.

Recipes
-------
* i.i.d. N(0,1): ``numpy.random.default_rng(seed).standard_normal`` in float32,
  drawn in the order Q, K, V, dO, then rounded to bf16/fp16 (round to nearest
  even, done by torch's CPU cast).
* Outlier distribution (FP8 accuracy protocol of the FlashAttention-3 paper,
  zenmind summary §10.3 / Table 3): N(0,1) where a Bernoulli(0.001) subset of
  entries is replaced by N(0, 10^2); with ``additive=True`` the N(0, 10^2)
  draw is added to those entries instead (the paper's own wording of the
  protocol), from the same random draws.
* Variable-length packing: sequence lengths drawn uniformly from [lo, hi] with
  ``integers(lo, hi + 1, n)``; ``cu_seqlens`` is their exclusive prefix sum.
* Random signs for the incoherent-processing rotation: +-1 drawn from the seed.
* Device-drawn N(0,1) for tensors too large to draw on the host in a test's
  time (past 2^31 elements): torch's seeded CUDA generator, drawn in the
  input dtype in the order of ``shapes``. Its values depend on torch's
  generator, not on this seed alone, so both sides of a comparison take the
  same drawn tensors (the oracle receives host copies of what it checks).
"""
from __future__ import annotations

import numpy as np
import torch

_TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def normal(seed: int, shapes, dtype: str = "bf16"):
    """Draw one tensor per entry of ``shapes`` (in order) from N(0,1).

    Returns CPU torch tensors of ``dtype`` ("bf16", "fp16" or "fp32").
    """
    rng = np.random.default_rng(seed)
    out = []
    for shp in shapes:
        x = rng.standard_normal(size=tuple(shp), dtype=np.float32)
        out.append(torch.from_numpy(x).to(_TORCH_DTYPES[dtype]))
    return out


def outliers(seed: int, shapes, dtype: str = "bf16", frac: float = 1e-3, sigma: float = 10.0,
             additive: bool = False):
    """N(0,1) with a Bernoulli(frac) subset of entries replaced by N(0, sigma^2)
    (``additive``: with N(0, sigma^2) added to them)."""
    rng = np.random.default_rng(seed)
    out = []
    for shp in shapes:
        x = rng.standard_normal(size=tuple(shp), dtype=np.float32)
        hit = rng.random(size=tuple(shp)) < frac
        extra = (sigma * rng.standard_normal(size=int(hit.sum()))).astype(np.float32)
        x[hit] = x[hit] + extra if additive else extra
        out.append(torch.from_numpy(x).to(_TORCH_DTYPES[dtype]))
    return out


def varlen_lengths(seed: int = 18, n: int = 8, lo: int = 1024, hi: int = 32768):
    """Sequence lengths drawn uniformly from the closed range [lo, hi]."""
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, n)]


def cu_seqlens(lengths):
    """Exclusive prefix sum of the lengths as an int32 tensor of size n+1."""
    c = np.zeros(len(lengths) + 1, dtype=np.int32)
    c[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return torch.from_numpy(c)


def random_signs(seed: int, d: int):
    """A vector of d random signs (+1/-1) as int8."""
    s = np.random.default_rng(seed).integers(0, 2, d)
    return torch.from_numpy((2 * s - 1).astype(np.int8))


def normal_device(seed: int, shapes, dtype: str = "bf16", device: str = "cuda"):
    """Draw one tensor per entry of ``shapes`` from N(0,1) on ``device``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return [torch.randn(tuple(shp), generator=gen, dtype=_TORCH_DTYPES[dtype], device=device) for shp in shapes]
