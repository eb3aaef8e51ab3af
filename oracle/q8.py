"""Q8 weights for the trimmed draft head: oracle (test infrastructure).

What the path computes (Small-vocabulary MTP study, section 3.3: the trimmed 32,768-row draft
head is served quantised -- its table compares a Q8 head with NVFP4 and a Q4_0 block; the
ShiftAddQwen README names the llama.cpp Q8_0 recipe among its baselines).  Q8 is read as that
recipe's plain definition: every 32 consecutive weights of a row along K share one fp16 scale
d, and each weight is an 8-bit two's-complement integer q, so

    w[n][k] = d[n][k // 32] * q[n][k].

Canonical inputs: codes int8 [N][K], scales fp16 bits [N][K/32].  The draft step is the
NVFP4 one (``oracle.nvfp4.draft_ids``): logits in fp64, argmax with the lowest row on ties,
mapped through the id map.

Packed layout (this project's kernel layout, restated from its written description):
  header as for INT4 (see ``oracle.int4``) with format 5, group 128, block bytes 17408.
  payload: row tiles of 128 (padding rows: codes 0 and scales 0).  Tile t and group g (inputs
    128g .. 128g+127) own one contiguous block of 17408 bytes at (t*(K/128) + g)*17408:
      codes: for 16-input chunk c = 0..7 and row r = n mod 128, the 16 code bytes of
        k = 128g + 16c .. +15 (in order) at c*2048 + r*16;
      scales: the fp16 bits of d[n][4g + j] at 16384 + j*256 + r*2 (j = 0..3).
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, f16_to_f64
from .int4 import HEADER_BYTES, MAGIC, ROW_TILE, GROUP, VERSION, parse_header

FORMAT_Q8 = 5
SUB = 32                                   # weights per fp16 scale
BLOCK_BYTES = 8 * ROW_TILE * 16 + 4 * ROW_TILE * 2


def dequant(codes: np.ndarray, scales_bits: np.ndarray) -> np.ndarray:
    """W[n][k] = d[n][k // 32] * q[n][k] in fp64."""
    q = np.asarray(codes, dtype=np.int8).astype(np.float64)
    d = f16_to_f64(scales_bits)
    N, K = q.shape
    assert K % SUB == 0 and d.shape == (N, K // SUB)
    return np.repeat(d, SUB, axis=1) * q


def gemm(x_bits: np.ndarray, codes: np.ndarray, scales_bits: np.ndarray,
         rows_per_block: int = 8192) -> np.ndarray:
    """Y64[m][n] = sum_k X[m][k] * W[n][k] (X as bf16 bits [M][K])."""
    X = bf16_to_f64(np.atleast_2d(x_bits))
    N = codes.shape[0]
    Y = np.empty((X.shape[0], N), dtype=np.float64)
    for n0 in range(0, N, rows_per_block):
        n1 = min(N, n0 + rows_per_block)
        Y[:, n0:n1] = X @ dequant(codes[n0:n1], scales_bits[n0:n1]).T
    return Y


# ----------------------------------------------------------------------------- layout

def packed_sizes(N: int, K: int):
    """(total bytes, payload offset, payload bytes, block bytes)."""
    NT = -(-N // ROW_TILE)
    payload = NT * (K // GROUP) * BLOCK_BYTES
    return HEADER_BYTES + payload, HEADER_BYTES, payload, BLOCK_BYTES


def header_bytes(N: int, K: int, payload: int) -> np.ndarray:
    h = np.zeros(HEADER_BYTES, dtype=np.uint8)
    h[0:32] = np.array([MAGIC, FORMAT_Q8, VERSION, N, K, 0, GROUP, ROW_TILE], dtype="<u4").view(np.uint8)
    h[32:64] = np.array([HEADER_BYTES, payload, BLOCK_BYTES, 0], dtype="<u8").view(np.uint8)
    return h


def pack(codes: np.ndarray, scales_bits: np.ndarray) -> np.ndarray:
    """Canonical codes int8 [N][K] and fp16 scale bits [N][K/32] -> packed bytes."""
    N, K = codes.shape
    G = K // GROUP
    assert K % GROUP == 0 and scales_bits.shape == (N, K // SUB)
    total, off, payload, blk = packed_sizes(N, K)
    NT = -(-N // ROW_TILE)
    Np = NT * ROW_TILE
    c = np.zeros((Np, K), dtype=np.uint8)
    c[:N] = np.asarray(codes, dtype=np.int8).view(np.uint8)
    # c[t*128 + r][128g + 16ch + b] -> [t][g][ch][r][b]
    c = np.ascontiguousarray(c.reshape(NT, ROW_TILE, G, 8, 16).transpose(0, 2, 3, 1, 4))
    d = np.zeros((Np, K // SUB), dtype=np.uint16)
    d[:N] = scales_bits
    d = np.ascontiguousarray(d.reshape(NT, ROW_TILE, G, 4).transpose(0, 2, 3, 1)).astype("<u2")  # [t][g][j][r]
    blocks = np.zeros((NT, G, blk), dtype=np.uint8)
    blocks[:, :, :16384] = c.reshape(NT, G, 16384)
    blocks[:, :, 16384:] = d.view(np.uint8).reshape(NT, G, 1024)
    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = header_bytes(N, K, payload)
    out[off:] = blocks.reshape(-1)
    return out


def unpack(packed: np.ndarray):
    """Packed bytes -> (codes int8 [N][K], scale bits uint16 [N][K/32])."""
    hd = parse_header(packed)
    assert hd["magic"] == MAGIC and hd["format"] == FORMAT_Q8 and hd["version"] == VERSION
    N, K = hd["N"], hd["K"]
    G = K // GROUP
    NT = -(-N // ROW_TILE)
    blocks = np.ascontiguousarray(
        packed[hd["payload_offset"]:hd["payload_offset"] + hd["payload_bytes"]]).reshape(NT, G, BLOCK_BYTES)
    c = blocks[:, :, :16384].reshape(NT, G, 8, ROW_TILE, 16).transpose(0, 3, 1, 2, 4)
    codes = np.ascontiguousarray(c.reshape(NT * ROW_TILE, K)[:N]).view(np.int8)
    d = np.ascontiguousarray(blocks[:, :, 16384:]).view("<u2").reshape(NT, G, 4, ROW_TILE).transpose(0, 3, 1, 2)
    scales = np.ascontiguousarray(d.reshape(NT * ROW_TILE, K // SUB)[:N]).astype(np.uint16)
    return codes, scales
