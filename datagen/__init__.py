"""Seeded synthetic inputs for the collective workloads.

This module holds no arithmetic of the collectives: it only draws numbers and
converts them to the storage dtype with library casts.  Both the oracle side
(tests, CPU baseline) and the CUDA side (tests, benchmark) take their inputs
from here.

Recipe: one fresh ``numpy.random.default_rng(seed)`` (PCG64) per workload and
dtype; ranks are drawn in rank order from that single stream.

* ``uniform``  : ``2 * rng.random(n, float32) - 1`` (uniform on [-1, 1), exact in f32)
* ``normal``   : ``rng.standard_normal(n, float32)``
* ``int``      : ``rng.integers(-1000, 1001, n)`` as int32 (uniform on [-1000, 1000])

f32 draws are cast to bf16 by ``torch.Tensor.to(torch.bfloat16)`` and to f16
by ``numpy.ndarray.astype(numpy.float16)`` (both round to nearest even).  bf16
values are stored as their uint16 bit patterns, f16 as uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

F32, BF16, F16, I32 = 0, 1, 2, 3
NAMES = {"f32": F32, "bf16": BF16, "f16": F16, "i32": I32}
STORAGE = {F32: np.float32, BF16: np.uint16, F16: np.uint16, I32: np.int32}
ESIZE = {F32: 4, BF16: 2, F16: 2, I32: 4}


def _cast(x32: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return x32
    if dtype == F16:
        return x32.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(dtype)


def draw(rng: np.random.Generator, dist: str, n: int, dtype: int) -> np.ndarray:
    if dist == "int":
        v = rng.integers(-1000, 1001, n)
        if dtype == I32:
            return v.astype(np.int32)
        return _cast(v.astype(np.float32), dtype)
    if dist == "uniform":
        x = 2 * rng.random(n, dtype=np.float32) - 1
    elif dist == "normal":
        x = rng.standard_normal(n, dtype=np.float32)
    elif dist == "smallint":
        # integers in [-4, 4]: every partial sum of up to 32 of them is an
        # exactly representable small integer in every dtype
        x = rng.integers(-4, 5, n).astype(np.float32)
    else:
        raise ValueError(dist)
    if dtype == I32:
        raise ValueError("int32 workloads draw from dist='int'")
    return _cast(x, dtype)


def rank_inputs(seed: int, dist: str, nranks: int, n: int, dtype: int):
    """``nranks`` arrays of ``n`` elements from one fresh generator."""
    rng = np.random.default_rng(seed)
    return [draw(rng, dist, n, dtype) for _ in range(nranks)]


def to_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of stored values to float64 (for tolerance checks)."""
    if dtype == F32:
        return a.astype(np.float64)
    if dtype == I32:
        return a.astype(np.float64)
    if dtype == F16:
        return a.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def alltoallv_counts(seed: int, nranks: int, tokens_per_rank: int, skew: float = 1.2) -> np.ndarray:
    """Token routing of a mixture-of-experts layer with one expert per rank:
    expert popularity follows a Zipf law of exponent ``skew`` over a random
    order of the experts (fresh generator from ``seed``), and every rank
    draws the destinations of its ``tokens_per_rank`` tokens from it
    (multinomial).  Returns counts[s][d] (int32, rows sum to
    tokens_per_rank)."""
    rng = np.random.default_rng(seed)
    weight = 1.0 / np.arange(1, nranks + 1, dtype=np.float64) ** skew
    p = weight[rng.permutation(nranks)]
    p /= p.sum()
    return np.stack([rng.multinomial(tokens_per_rank, p) for _ in range(nranks)]).astype(np.int32)
