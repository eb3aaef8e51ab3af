"""Storage-type decoding and bf16 rounding for the oracle (test infrastructure).

The pages fix the storage types: 16-bit activations (the W4A16 format of the Efficient-Qwen
report, section 2.1), fp16 per-group scales.  Outputs are bf16, rounded once from the exact
(fp64) result with round-to-nearest, ties-to-even.
"""
from __future__ import annotations

import numpy as np


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """IEEE fp16 bit patterns (uint16) -> fp64 values (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64 values (exact: bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even; returns fp64 values.

    bf16 carries 8 significant bits.  Write x = m * 2**e with 0.5 <= |m| < 1; the bf16
    neighbours of x are multiples of 2**(e-8), so x rounds to rint(m * 2**8) * 2**(e-8)
    (numpy's rint rounds halves to even).  Below bf16's normal range the spacing stays
    2**-133.  Values beyond the largest finite bf16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    e = np.maximum(e, -125)          # subnormal spacing 2**-133 = 2**(-125-8)
    r = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    big = np.abs(r) >= 2.0 ** 128
    return np.where(big, np.copysign(np.inf, x), r)


def bf16_bits(x_rounded: np.ndarray) -> np.ndarray:
    """bf16-representable fp64 values -> uint16 bit patterns."""
    f = np.asarray(x_rounded, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
