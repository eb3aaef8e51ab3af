"""NVFP4 weights and the trimmed draft head: oracle (test infrastructure).

What the path computes (Small-vocabulary MTP study, abstract and section 3.3: trim the draft
head to the model's own 32,768 most used tokens, quantise it to NVFP4, and map each draft
row back to its full-vocabulary token id before verifying against the full vocabulary).

NVFP4 (the public format the study names): each weight is a 4-bit E2M1 float -- sign bit,
two exponent bits with bias 1, one mantissa bit, so the magnitudes are
    e = 0: m * 0.5               (0, 0.5)
    e > 0: 2^(e-1) * (1 + m/2)   (1, 1.5, 2, 3, 4, 6)
-- every 16 consecutive weights of a row along K share one FP8 E4M3 scale (sign, four
exponent bits with bias 7, three mantissa bits; exponent 0 is subnormal, m * 2^-9; the code
0x7F / 0xFF is NaN and there is no infinity), and the tensor has one fp32 scale:

    w[n][k] = g * e4m3(s[n][k // 16]) * e2m1(c[n][k]).

Canonical inputs: codes uint8 [N][K/2] (element k in byte k // 2, the low nibble for even k),
scales uint8 [N][K/16] (E4M3 bits), g a float.

The draft step: logits[m][n] = sum_k h[m][k] * w[n][k] (fp64 here), a[m] = argmax_n with the
lowest row on ties, and the emitted id is id_map[a[m]] (a[m] itself when there is no map).

Packed layout (this project's kernel layout, restated from its written description):
  header as for INT4 (see ``oracle.int4``) with format 4, group 128, block bytes 9216, and
    the fp32 bits of g in the low 4 bytes of the final u64 field (byte offset 56).
  payload: row tiles of 128 (padding rows: codes 0 and scales 0).  Tile t and group g (inputs
    128g .. 128g+127) own one contiguous block of 9216 bytes at (t*(K/128) + g)*9216:
      codes: for 32-input chunk c = 0..3 and row r = n mod 128, the 16 canonical code bytes
        of k = 128g + 32c .. +31 at c*2048 + r*16;
      scales: the E4M3 byte of s[n][8g + j] at 8192 + j*128 + r (j = 0..7).
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64
from .int4 import HEADER_BYTES, MAGIC, ROW_TILE, GROUP, VERSION, parse_header

FORMAT_NVFP4 = 4
SUB = 16                                   # weights per E4M3 scale
BLOCK_BYTES = 4 * ROW_TILE * 16 + 8 * ROW_TILE


def e2m1_to_f64(codes: np.ndarray) -> np.ndarray:
    """4-bit E2M1 codes (0..15) -> fp64, from the field definitions."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return sign * mag


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bytes -> fp64, from the field definitions (0x7F / 0xFF are NaN)."""
    b = np.asarray(bits, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 15
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, np.ldexp(m, -9), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((b & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [N][K/2] -> 4-bit codes [N][K] (low nibble = even element)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = c & 15
    out[..., 1::2] = c >> 4
    return out


def dequant(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """W[n][k] = g * e4m3(s[n][k // 16]) * e2m1(c[n][k]) in fp64."""
    q = e2m1_to_f64(unpack_codes(codes))
    N, K = q.shape
    s = e4m3_to_f64(scales)
    assert K % SUB == 0 and s.shape == (N, K // SUB)
    return float(np.float32(g)) * np.repeat(s, SUB, axis=1) * q


def gemm(x_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, g: float,
         rows_per_block: int = 8192) -> np.ndarray:
    """logits64[m][n] = sum_k X[m][k] * W[n][k] (X as bf16 bits [M][K])."""
    X = bf16_to_f64(np.atleast_2d(x_bits))
    N = codes.shape[0]
    Y = np.empty((X.shape[0], N), dtype=np.float64)
    for n0 in range(0, N, rows_per_block):
        n1 = min(N, n0 + rows_per_block)
        Y[:, n0:n1] = X @ dequant(codes[n0:n1], scales[n0:n1], g).T
    return Y


def draft_ids(logits: np.ndarray, id_map: np.ndarray | None = None) -> np.ndarray:
    """Per row of logits: the lowest-indexed maximum, mapped through id_map when given."""
    from .verify import argmax_lowest
    a = argmax_lowest(np.atleast_2d(logits))
    return a if id_map is None else np.asarray(id_map)[a]


# ----------------------------------------------------------------------------- layout

def packed_sizes(N: int, K: int):
    """(total bytes, payload offset, payload bytes, block bytes)."""
    NT = -(-N // ROW_TILE)
    payload = NT * (K // GROUP) * BLOCK_BYTES
    return HEADER_BYTES + payload, HEADER_BYTES, payload, BLOCK_BYTES


def header_bytes(N: int, K: int, payload: int, g: float) -> np.ndarray:
    h = np.zeros(HEADER_BYTES, dtype=np.uint8)
    h[0:32] = np.array([MAGIC, FORMAT_NVFP4, VERSION, N, K, 0, GROUP, ROW_TILE], dtype="<u4").view(np.uint8)
    gbits = int(np.array([g], dtype="<f4").view("<u4")[0])
    h[32:64] = np.array([HEADER_BYTES, payload, BLOCK_BYTES, gbits], dtype="<u8").view(np.uint8)
    return h


def pack(codes: np.ndarray, scales: np.ndarray, g: float) -> np.ndarray:
    """Canonical codes uint8 [N][K/2], E4M3 scales uint8 [N][K/16], g -> packed bytes."""
    N, KB = codes.shape
    K = KB * 2
    G = K // GROUP
    assert K % GROUP == 0 and scales.shape == (N, K // SUB)
    total, off, payload, blk = packed_sizes(N, K)
    NT = -(-N // ROW_TILE)
    Np = NT * ROW_TILE
    c = np.zeros((Np, KB), dtype=np.uint8)
    c[:N] = codes
    # c[t*128 + r][64g + 16ch + b] -> [t][g][ch][r][b]
    c = np.ascontiguousarray(c.reshape(NT, ROW_TILE, G, 4, 16).transpose(0, 2, 3, 1, 4))
    s = np.zeros((Np, K // SUB), dtype=np.uint8)
    s[:N] = scales
    s = np.ascontiguousarray(s.reshape(NT, ROW_TILE, G, 8).transpose(0, 2, 3, 1))   # [t][g][j][r]
    blocks = np.zeros((NT, G, blk), dtype=np.uint8)
    blocks[:, :, :8192] = c.reshape(NT, G, 8192)
    blocks[:, :, 8192:] = s.reshape(NT, G, 1024)
    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = header_bytes(N, K, payload, g)
    out[off:] = blocks.reshape(-1)
    return out


def unpack(packed: np.ndarray):
    """Packed bytes -> (codes uint8 [N][K/2], scales uint8 [N][K/16], g)."""
    hd = parse_header(packed)
    assert hd["magic"] == MAGIC and hd["format"] == FORMAT_NVFP4 and hd["version"] == VERSION
    N, K = hd["N"], hd["K"]
    G = K // GROUP
    NT = -(-N // ROW_TILE)
    g = float(np.asarray(packed[56:60], dtype=np.uint8).view("<f4")[0])
    blocks = np.ascontiguousarray(
        packed[hd["payload_offset"]:hd["payload_offset"] + hd["payload_bytes"]]).reshape(NT, G, BLOCK_BYTES)
    c = blocks[:, :, :8192].reshape(NT, G, 4, ROW_TILE, 16).transpose(0, 3, 1, 2, 4)
    codes = np.ascontiguousarray(c.reshape(NT * ROW_TILE, K // 2)[:N])
    s = blocks[:, :, 8192:].reshape(NT, G, 8, ROW_TILE).transpose(0, 3, 1, 2)
    scales = np.ascontiguousarray(s.reshape(NT * ROW_TILE, K // SUB)[:N])
    return codes, scales, g
