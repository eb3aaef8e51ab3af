"""ShiftAdd binary-plane weights: oracle (test infrastructure).

What the path computes (ShiftAddQwen README, introduction and "Method"/"Format"): each
weight group is a sum of binary planes with per-group scales,

    w[n][k] = sum_p alpha[p][n][k // G] * b[p][n][k],   b in {-1, +1},

so a mat-vec is, per plane, a sign-select-and-add over the group followed by one scale per
group.  Here the scale is one fp16 alpha per (plane, row, group of G = 128 inputs); the
product is computed exactly in fp64 and rounded once to bf16.

Canonical sign-bit input: uint8 [P][N][K/8]; bit j (LSB first) of byte i is element
k = 8i + j, and a set bit means +1.

Packed layout (this project's kernel layout, restated from its written description):
  header as for INT4 (see ``oracle.int4``) with format 2, P planes and block bytes 2304*P.
  payload: row tiles of 128 (padding rows: all bits 0 and alpha 0).  Tile t and group g own
    one contiguous block of 2304*P bytes at (t*(K/128) + g)*2304*P:
      signs: for plane p and row r = n mod 128, 16 bytes at p*2048 + r*16 holding the 128
        sign bits of k = 128g .. 128g+127 as four little-endian u32 words.  Word w covers
        k0 = 128g + 32w: bit i (i = 0..15) is the sign of k0 + 2i and bit 16 + i the sign of
        k0 + 2i + 1 (even inputs in the low half-word, odd inputs in the high half-word);
      alphas: fp16 bits of alpha[p][n][g] at 2048*P + (p*128 + r)*2.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, f16_to_f64
from .int4 import HEADER_BYTES, MAGIC, ROW_TILE, GROUP, VERSION, header_bytes, parse_header

FORMAT_BINPLANE = 2


def signs(bits: np.ndarray) -> np.ndarray:
    """uint8 [P][N][K/8] sign bits -> fp64 [P][N][K] with values +1 (bit set) or -1."""
    b = np.unpackbits(np.asarray(bits, dtype=np.uint8), axis=-1, bitorder="little")
    return np.where(b == 1, 1.0, -1.0)


def dequant(bits: np.ndarray, alpha_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """W[n][k] = sum_p alpha[p][n][k // group] * b[p][n][k] in fp64."""
    b = signs(bits)                              # [P][N][K]
    a = f16_to_f64(alpha_bits)                   # [P][N][K/group]
    P, N, K = b.shape
    assert K % group == 0 and a.shape == (P, N, K // group)
    return np.sum(np.repeat(a, group, axis=2) * b, axis=0)


def gemm(x_bits: np.ndarray, bits: np.ndarray, alpha_bits: np.ndarray,
         group: int = GROUP, rows_per_block: int = 4096) -> np.ndarray:
    """Y64[m][n] = sum_k X[m][k] * W[n][k] in fp64 (blocks of output rows bound memory)."""
    X = bf16_to_f64(np.atleast_2d(x_bits))
    N = bits.shape[1]
    Y = np.empty((X.shape[0], N), dtype=np.float64)
    for n0 in range(0, N, rows_per_block):
        n1 = min(N, n0 + rows_per_block)
        Y[:, n0:n1] = X @ dequant(bits[:, n0:n1], alpha_bits[:, n0:n1], group).T
    return Y


# ----------------------------------------------------------------------------- layout

def block_bytes(P: int) -> int:
    return P * (ROW_TILE * 16 + ROW_TILE * 2)


def packed_sizes(P: int, N: int, K: int):
    """(total bytes, payload offset, payload bytes, block bytes)."""
    NT = -(-N // ROW_TILE)
    payload = NT * (K // GROUP) * block_bytes(P)
    return HEADER_BYTES + payload, HEADER_BYTES, payload, block_bytes(P)


def pack(bits: np.ndarray, alpha_bits: np.ndarray) -> np.ndarray:
    """Canonical sign bits [P][N][K/8] and fp16 alphas [P][N][K/128] -> packed bytes."""
    P, N, KB = bits.shape
    K = KB * 8
    G = K // GROUP
    assert K % GROUP == 0 and alpha_bits.shape == (P, N, G)
    total, off, payload, blk = packed_sizes(P, N, K)
    NT = -(-N // ROW_TILE)
    Np = NT * ROW_TILE
    beta = np.zeros((P, Np, K), dtype=np.uint32)
    beta[:, :N] = np.unpackbits(bits, axis=-1, bitorder="little")
    # beta[p][t*128 + r][128g + 32w + 2i + o] -> axes [p][t][r][g][w][i][o]
    b7 = beta.reshape(P, NT, ROW_TILE, G, 4, 16, 2)
    shift = (np.arange(16, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])          # [i][o]
    words = np.bitwise_or.reduce(
        np.bitwise_or.reduce(b7 << shift, axis=6), axis=5)            # [p][t][r][g][w]
    words = np.ascontiguousarray(words.transpose(1, 3, 0, 2, 4)).astype("<u4")  # [t][g][p][r][w]
    a = np.zeros((P, Np, G), dtype=np.uint16)
    a[:, :N] = alpha_bits
    a = np.ascontiguousarray(a.reshape(P, NT, ROW_TILE, G).transpose(1, 3, 0, 2)).astype("<u2")  # [t][g][p][r]
    blocks = np.zeros((NT, G, blk), dtype=np.uint8)
    blocks[:, :, :2048 * P] = words.reshape(NT, G, 512 * P).view(np.uint8)
    blocks[:, :, 2048 * P:] = a.view(np.uint8).reshape(NT, G, 256 * P)
    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = header_bytes(FORMAT_BINPLANE, N, K, P, payload, blk)
    out[off:] = blocks.reshape(-1)
    return out


def unpack(packed: np.ndarray):
    """Packed bytes -> (sign bits uint8 [P][N][K/8], fp16 alpha bits [P][N][K/128])."""
    hd = parse_header(packed)
    assert hd["magic"] == MAGIC and hd["format"] == FORMAT_BINPLANE and hd["version"] == VERSION
    P, N, K = hd["P"], hd["N"], hd["K"]
    G = K // GROUP
    NT = -(-N // ROW_TILE)
    blocks = np.ascontiguousarray(
        packed[hd["payload_offset"]:hd["payload_offset"] + hd["payload_bytes"]]
    ).reshape(NT, G, block_bytes(P))
    words = np.ascontiguousarray(blocks[:, :, :2048 * P]).view("<u4").reshape(NT, G, P, ROW_TILE, 4)
    shift = (np.arange(16, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])
    b = (words[..., None, None] >> shift) & np.uint32(1)             # [t][g][p][r][w][i][o]
    b = b.transpose(2, 0, 3, 1, 4, 5, 6).reshape(P, NT * ROW_TILE, K)[:, :N]
    bits = np.packbits(b.astype(np.uint8), axis=-1, bitorder="little")
    a = np.ascontiguousarray(blocks[:, :, 2048 * P:]).view("<u2").reshape(NT, G, P, ROW_TILE)
    a = a.transpose(2, 0, 3, 1)
    alpha = np.ascontiguousarray(a.reshape(P, NT * ROW_TILE, G)[:, :N]).astype(np.uint16)
    return bits, alpha
