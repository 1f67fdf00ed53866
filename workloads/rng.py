"""Seeded value sources for the synthetic workloads.

This module draws numbers and encodes them as bf16 bit patterns. It holds none
of the attention, paging or allocation arithmetic: both the GPU path (through
the Python binding) and the CPU oracle receive the arrays it returns as plain
inputs.

Values are N(0, 1) draws from numpy's PCG64 generator, keyed by an integer
seed, rounded first to float32 and then to bf16 (round to nearest even).
"""

from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as bf16 bit patterns, round to nearest even.

    Inputs are finite draws; NaN/Inf handling is not needed here.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
            >> np.uint32(16)).astype(np.uint16)


def generator(*key: int) -> np.random.Generator:
    """A PCG64 generator keyed by a tuple of non-negative integers."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def normal_bf16_from(g: np.random.Generator, shape, chunk: int = 1 << 26) -> np.ndarray:
    """Draw N(0,1) values from ``g`` as bf16 bits (uint16 array of ``shape``)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        out[lo:hi] = f32_to_bf16_bits(g.standard_normal(hi - lo, dtype=np.float32))
    return out.reshape(shape)


def normal_bf16(shape, *key: int) -> np.ndarray:
    """N(0,1) values as bf16 bits from a fresh generator keyed by ``key``."""
    return normal_bf16_from(generator(*key), shape)


# bf16 bit pattern of a quiet NaN, used to poison cache slots that no sequence owns.
BF16_NAN = np.uint16(0x7FC0)
