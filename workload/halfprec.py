"""16-bit copies of input values (bfloat16 and IEEE binary16 bit patterns).

Input preparation only, for the reduced-precision host values of the host
pass: rounding float32 values to 16 bits and reading them back.  No cosine
arithmetic here.
"""
from __future__ import annotations

import numpy as np


def to_bf16_bits(values: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns of finite float32 values, rounded to nearest, ties to even."""
    u = np.ascontiguousarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """The float32 values of bfloat16 bit patterns (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_f16_bits(values: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns of float32 values (numpy's round to nearest even)."""
    return np.ascontiguousarray(values, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """The float32 values of binary16 bit patterns (exact)."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


# Unit roundoff of round-to-nearest conversion to each format.
UNIT_ROUNDOFF = {"bf16": 2.0 ** -9, "f16": 2.0 ** -11}
