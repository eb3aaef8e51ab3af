"""Shared test helpers: device transfer and the parity criteria.

Parity criteria (the bar every GPU result is held to):
  * packing and acceptance: bit-exact;
  * GEMM outputs: |gpu - RNE_bf16(Y64)| <= 1e-2 * rms(oracle row) + 1e-3, where an output
    whose exact value lies within a small band around the midpoint of two bf16 neighbours may
    take either neighbour (bf16 rounding is a decision on a value the two sides compute in
    different precisions);
  * argmax: equal wherever the oracle's top-1 margin exceeds 1e-2, otherwise the GPU's row
    must be a valid near-maximum (its oracle logit within 1e-2 of the maximum).
"""
from __future__ import annotations

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import numerics  # noqa: E402

REL_TOL = 1e-2
ABS_TOL = 1e-3
MARGIN = 1e-2


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits):
    import torch
    return dev(bits.view(np.int16), torch.bfloat16) if bits.dtype == np.uint16 else dev(bits)


def f16_dev(bits):
    import torch
    return dev(bits.view(np.int16), torch.float16)


def host_bits(t):
    """Device bf16/fp16 tensor -> numpy uint16 bits."""
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_gemm(y_gpu_bits: np.ndarray, Y64: np.ndarray, what: str = "", scale: float = 1.0):
    """Assert the GEMM parity criterion; returns (max normalised error, boundary cases).

    ``scale`` (a power of two) multiplies both sides before the comparison, so outputs of
    inputs drawn at 2^-90 or 2^90 are held to the same relative bar; bf16 rounding commutes
    with it while the values stay normal."""
    Y64 = np.atleast_2d(Y64)
    r = numerics.round_to_bf16(Y64) * scale
    g = numerics.bf16_to_f64(np.atleast_2d(y_gpu_bits)) * scale
    Y64 = Y64 * scale
    rms = np.sqrt(np.mean(Y64 ** 2, axis=1, keepdims=True))
    tol = REL_TOL * rms + ABS_TOL
    err = np.abs(g - r)
    bad = err > tol
    n_boundary = 0
    if bad.any():
        # admissible only if the GPU value is the other bf16 neighbour of Y64 and Y64 sits in
        # a band of 1e-3 * rms + 1e-4 around the rounding midpoint of the two neighbours.
        band = (1e-3 * rms + 1e-4) * np.ones_like(Y64)
        mid = 0.5 * (g + r)
        neighbour = np.abs(g - Y64) < np.abs(g - r) + 1e-300
        near_mid = np.abs(Y64 - mid) <= band
        ok = neighbour & near_mid
        n_boundary = int((bad & ok).sum())
        # Such cases need the GPU's value and the exact one on either side of a midpoint
        # within the band: rare for any kernel whose error is far below the tolerance.
        assert n_boundary <= max(4, Y64.size // 10000), \
            f"{what}: {n_boundary} outputs on the other side of a bf16 rounding midpoint"
        still = bad & ~ok
        if still.any():
            idx = np.argwhere(still)[:5]
            raise AssertionError(
                f"{what}: {int(still.sum())} outputs outside tolerance, e.g. "
                + ", ".join(f"[{m},{n}] gpu={g[m, n]!r} oracle={Y64[m, n]!r} tol={tol[m, 0]:.3g}"
                            for m, n in idx))
    return float(np.max(err / tol)), n_boundary


def check_argmax(a_gpu: np.ndarray, logits64: np.ndarray, what: str = ""):
    """Argmax criterion; returns the number of rows graded only as near-ties."""
    from oracle import verify
    a_ref = verify.argmax_lowest(logits64)
    margin = verify.top2_margin(logits64)
    ungraded = 0
    for m in range(logits64.shape[0]):
        if margin[m] > MARGIN:
            assert a_gpu[m] == a_ref[m], f"{what}: row {m} gpu {a_gpu[m]} oracle {a_ref[m]}"
        else:
            ungraded += 1
            assert 0 <= a_gpu[m] < logits64.shape[1]
            assert logits64[m, a_gpu[m]] >= logits64[m, a_ref[m]] - MARGIN, what
    return ungraded


class Guarded:
    """A device tensor with canary bands on both sides: ``t`` is the view a call writes; the
    bands (``band`` elements each side) hold a fixed byte pattern that ``check()`` asserts
    is unchanged, so a write past either end of the output is caught."""

    PATTERN = 0xA5

    def __init__(self, shape, dtype, band=256, fill=None):
        import torch
        n = 1
        for d in shape:
            n *= d
        self.band, self.n = band, n
        self.buf = torch.empty(n + 2 * band, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(self.PATTERN)
        self.t = self.buf[band:band + n].view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what=""):
        import torch
        b = self.buf.view(torch.uint8).cpu().numpy()
        es = self.buf.element_size()
        lo, hi = b[:self.band * es], b[(self.band + self.n) * es:]
        assert (lo == self.PATTERN).all() and (hi == self.PATTERN).all(), f"{what}: canary overwritten"
