"""Symmetric per-group INT4 weights: oracle (test infrastructure).

What the path computes (Efficient-Qwen report, section 2.1 "Target Model Optimization with
QAD" and section 3.3 "Drafter PTQ"): the weight is W = s (.) W_q, INT4 codes q in [-8, 7]
with one symmetric scale s per group of 128 consecutive input features, served as W4A16
(16-bit activations).  A linear layer's output is then

    y[m][n] = sum_k x[m][k] * s[n][k // G] * q[n][k],

computed here exactly in fp64 and rounded once to bf16.  The group size G is a parameter so
the hand-worked examples can use G = 4 and G = 8; the library itself uses G = 128.

The packed byte layout (``pack``/``unpack``) is this project's kernel layout, restated here
from its written description, independently of the CUDA source:

  header (128 B, little-endian): u32 magic 0x3242574C, u32 format (1 = INT4),
    u32 version (2), u32 N, u32 K, u32 P (0 for INT4), u32 group (128), u32 row tile (128),
    u64 payload offset (128), u64 payload bytes, u64 block bytes (8448), u64 0, zero padding.
  payload: rows are grouped in tiles of 128 (N padded up to NT = ceil(N/128) tiles; padding
    rows hold q = 0 and scale 0).  Tile t and group g (inputs 128g .. 128g+127) own one
    contiguous block of 8448 bytes at (t*(K/128) + g)*8448:
      codes: for 32-input chunk c = 0..3 and row r = n mod 128, 16 bytes at c*2048 + r*16,
        four little-endian u32 words; word i holds k = 128g + 32c + 8i + 2p + o
        (p = 0..3, o = 0..1) as the nibble u = q + 8 at bit 4p + 16o;
      scales: fp16 bits of s[n][g] at 8192 + r*2.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, f16_to_f64

MAGIC = 0x3242574C
FORMAT_INT4 = 1
VERSION = 2
HEADER_BYTES = 128
ROW_TILE = 128
GROUP = 128
INT4_BLOCK_BYTES = 4 * ROW_TILE * 16 + ROW_TILE * 2      # 8192 code bytes + 256 scale bytes


def dequant(codes: np.ndarray, scales_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """W[n][k] = s[n][k // group] * q[n][k] in fp64."""
    q = np.asarray(codes, dtype=np.int64).astype(np.float64)
    s = f16_to_f64(scales_bits)
    N, K = q.shape
    assert K % group == 0 and s.shape == (N, K // group)
    return np.repeat(s, group, axis=1) * q


def gemm(x_bits: np.ndarray, codes: np.ndarray, scales_bits: np.ndarray,
         group: int = GROUP, rows_per_block: int = 8192) -> np.ndarray:
    """Y64[m][n] = sum_k X[m][k] * W[n][k] in fp64 (X given as bf16 bits [M][K]).

    Output rows are produced ``rows_per_block`` weight rows at a time only to bound the
    memory of the dequantised fp64 weights; every output is the same full dot product.
    """
    X = bf16_to_f64(np.atleast_2d(x_bits))
    N = codes.shape[0]
    Y = np.empty((X.shape[0], N), dtype=np.float64)
    for n0 in range(0, N, rows_per_block):
        n1 = min(N, n0 + rows_per_block)
        Y[:, n0:n1] = X @ dequant(codes[n0:n1], scales_bits[n0:n1], group).T
    return Y


# ----------------------------------------------------------------------------- layout

def packed_sizes(N: int, K: int):
    """(total bytes, payload offset, payload bytes, block bytes)."""
    NT = -(-N // ROW_TILE)
    payload = NT * (K // GROUP) * INT4_BLOCK_BYTES
    return HEADER_BYTES + payload, HEADER_BYTES, payload, INT4_BLOCK_BYTES


def header_bytes(fmt: int, N: int, K: int, P: int, payload: int, block: int) -> np.ndarray:
    h = np.zeros(HEADER_BYTES, dtype=np.uint8)
    u32 = np.array([MAGIC, fmt, VERSION, N, K, P, GROUP, ROW_TILE], dtype="<u4")
    u64 = np.array([HEADER_BYTES, payload, block, 0], dtype="<u8")
    h[0:32] = u32.view(np.uint8)
    h[32:64] = u64.view(np.uint8)
    return h


def pack(codes: np.ndarray, scales_bits: np.ndarray) -> np.ndarray:
    """Canonical codes int8 [N][K] and fp16 scales [N][K/128] -> packed bytes (uint8)."""
    N, K = codes.shape
    G = K // GROUP
    assert K % GROUP == 0 and scales_bits.shape == (N, G)
    total, off, payload, block = packed_sizes(N, K)
    NT = -(-N // ROW_TILE)
    Np = NT * ROW_TILE
    u = np.full((Np, K), 8, dtype=np.uint32)
    u[:N] = (np.asarray(codes, dtype=np.int32) + 8).astype(np.uint32)
    # u[t*128 + r][128g + 32c + 8i + 2p + o] -> axes [t][r][g][c][i][p][o]
    u7 = u.reshape(NT, ROW_TILE, G, 4, 4, 4, 2)
    shift = (4 * np.arange(4, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])          # [p][o]
    words = np.bitwise_or.reduce(
        np.bitwise_or.reduce(u7 << shift, axis=6), axis=5)            # [t][r][g][c][i]
    words = np.ascontiguousarray(words.transpose(0, 2, 3, 1, 4)).astype("<u4")  # [t][g][c][r][i]
    s = np.zeros((Np, G), dtype=np.uint16)
    s[:N] = scales_bits
    s = np.ascontiguousarray(s.reshape(NT, ROW_TILE, G).transpose(0, 2, 1)).astype("<u2")  # [t][g][r]
    blocks = np.zeros((NT, G, block), dtype=np.uint8)
    blocks[:, :, :8192] = words.reshape(NT, G, 8192 // 4).view(np.uint8)
    blocks[:, :, 8192:] = s.view(np.uint8).reshape(NT, G, 256)
    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = header_bytes(FORMAT_INT4, N, K, 0, payload, block)
    out[off:] = blocks.reshape(-1)
    return out


def parse_header(packed: np.ndarray) -> dict:
    h = np.asarray(packed[:HEADER_BYTES], dtype=np.uint8)
    u32 = h[0:32].view("<u4")
    u64 = h[32:64].view("<u8")
    return dict(magic=int(u32[0]), format=int(u32[1]), version=int(u32[2]), N=int(u32[3]),
                K=int(u32[4]), P=int(u32[5]), group=int(u32[6]), row_tile=int(u32[7]),
                payload_offset=int(u64[0]), payload_bytes=int(u64[1]), block_bytes=int(u64[2]))


def unpack(packed: np.ndarray):
    """Packed bytes -> (codes int8 [N][K], fp16 scale bits [N][K/128])."""
    hd = parse_header(packed)
    assert hd["magic"] == MAGIC and hd["format"] == FORMAT_INT4 and hd["version"] == VERSION
    N, K = hd["N"], hd["K"]
    G = K // GROUP
    NT = -(-N // ROW_TILE)
    blocks = np.ascontiguousarray(
        packed[hd["payload_offset"]:hd["payload_offset"] + hd["payload_bytes"]]
    ).reshape(NT, G, INT4_BLOCK_BYTES)
    words = np.ascontiguousarray(blocks[:, :, :8192]).view("<u4").reshape(NT, G, 4, ROW_TILE, 4)
    words = words.transpose(0, 3, 1, 2, 4)                            # [t][r][g][c][i]
    shift = (4 * np.arange(4, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])
    u = (words[..., None, None] >> shift) & np.uint32(0xF)          # [t][r][g][c][i][p][o]
    codes = (u.reshape(NT * ROW_TILE, K).astype(np.int16) - 8).astype(np.int8)[:N]
    s = np.ascontiguousarray(blocks[:, :, 8192:]).view("<u2").reshape(NT, G, ROW_TILE)
    scales = np.ascontiguousarray(s.transpose(0, 2, 1).reshape(NT * ROW_TILE, G)[:N]).astype(np.uint16)
    return codes, scales
