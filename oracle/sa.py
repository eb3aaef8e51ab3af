"""ShiftAdd binary planes with u8 scale codes (the deployed sa format): oracle (test
infrastructure).

What the path computes (ShiftAddQwen README, "Format"): along the input dimension the
weights of a row come in super-blocks of 256; a super-block stores Q sign planes, one u8 scale
code a per plane and group of G in {64, 128, 256} inputs, and one fp16 scale d, and the plane
scale is alpha = d * a.  With the plane sum of the README's introduction,

    w[n][k] = d[n][k // 256] * sum_p a[p][n][k // G] * b[p][n][k],   b in {-1, +1},

and a linear layer's output y[m][n] = sum_k x[m][k] * w[n][k], computed here exactly in
fp64 and rounded once to bf16.

Canonical inputs: sign bits uint8 [P][N][K/8] (bit j, LSB first, of byte i is element
k = 8i + j; a set bit means +1), codes uint8 [P][N][K/G], d as fp16 bits [N][K/256].

Packed layout (this project's kernel layout, restated from its written description):
  header as for INT4 (see ``oracle.int4``) with format 3, P planes, group G and block bytes
    B = 4096*P + 128*P*(256/G) + 256.
  payload: row tiles of 128 (padding rows: all bits 0, codes 0, d 0).  Tile t and super-block
    j (inputs 256j .. 256j+255) own one contiguous block of B bytes at (t*(K/256) + j)*B:
      signs: for plane p, half h = 0, 1 and row r = n mod 128, 16 bytes at
        p*4096 + h*2048 + r*16 holding four little-endian u32 words; word w covers
        k0 = 256j + 128h + 32w: bit i (i = 0..15) is the sign of k0 + 2i and bit 16 + i the
        sign of k0 + 2i + 1;
      codes: a[p][n][g] at 4096*P + (p*(256/G) + g - j*(256/G))*128 + r;
      d: fp16 bits of d[n][j] at 4096*P + 128*P*(256/G) + r*2.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, f16_to_f64
from .int4 import HEADER_BYTES, MAGIC, ROW_TILE, VERSION, parse_header
from .binplane import signs

FORMAT_SA = 3
SUPER = 256
GROUPS = (64, 128, 256)


def dequant(bits: np.ndarray, codes: np.ndarray, d_bits: np.ndarray, group: int) -> np.ndarray:
    """W[n][k] = d[n][k // 256] * sum_p a[p][n][k // group] * b[p][n][k] in fp64."""
    b = signs(bits)                                   # [P][N][K]
    a = np.asarray(codes, dtype=np.uint8).astype(np.float64)
    d = f16_to_f64(d_bits)
    P, N, K = b.shape
    assert K % SUPER == 0 and group in GROUPS
    assert a.shape == (P, N, K // group) and d.shape == (N, K // SUPER)
    plane_sum = np.sum(np.repeat(a, group, axis=2) * b, axis=0)      # sum_p a_p b_p, [N][K]
    return np.repeat(d, SUPER, axis=1) * plane_sum


def gemm(x_bits: np.ndarray, bits: np.ndarray, codes: np.ndarray, d_bits: np.ndarray,
         group: int, rows_per_block: int = 4096) -> np.ndarray:
    """Y64[m][n] = sum_k X[m][k] * W[n][k] in fp64 (blocks of output rows bound memory)."""
    X = bf16_to_f64(np.atleast_2d(x_bits))
    N = bits.shape[1]
    Y = np.empty((X.shape[0], N), dtype=np.float64)
    for n0 in range(0, N, rows_per_block):
        n1 = min(N, n0 + rows_per_block)
        Y[:, n0:n1] = X @ dequant(bits[:, n0:n1], codes[:, n0:n1], d_bits[n0:n1], group).T
    return Y


def gemm_entries(x_bits: np.ndarray, bits: np.ndarray, codes: np.ndarray, d_bits: np.ndarray,
                 group: int, rows: np.ndarray) -> np.ndarray:
    """Y64[:, rows] only (for sampled checks on large matrices)."""
    rows = np.asarray(rows)
    return gemm(x_bits, bits[:, rows], codes[:, rows], d_bits[rows], group)


# ----------------------------------------------------------------------------- layout

def block_bytes(P: int, group: int) -> int:
    return P * ROW_TILE * 32 + P * (SUPER // group) * ROW_TILE + ROW_TILE * 2


def packed_sizes(P: int, group: int, N: int, K: int):
    """(total bytes, payload offset, payload bytes, block bytes)."""
    NT = -(-N // ROW_TILE)
    blk = block_bytes(P, group)
    payload = NT * (K // SUPER) * blk
    return HEADER_BYTES + payload, HEADER_BYTES, payload, blk


def header_bytes(N: int, K: int, P: int, group: int, payload: int, block: int) -> np.ndarray:
    h = np.zeros(HEADER_BYTES, dtype=np.uint8)
    h[0:32] = np.array([MAGIC, FORMAT_SA, VERSION, N, K, P, group, ROW_TILE], dtype="<u4").view(np.uint8)
    h[32:64] = np.array([HEADER_BYTES, payload, block, 0], dtype="<u8").view(np.uint8)
    return h


def pack(bits: np.ndarray, codes: np.ndarray, d_bits: np.ndarray, group: int) -> np.ndarray:
    """Canonical sign bits [P][N][K/8], u8 codes [P][N][K/G] and fp16 d [N][K/256] -> packed
    bytes."""
    P, N, KB = bits.shape
    K = KB * 8
    J, GJ = K // SUPER, SUPER // group          # super-blocks, groups per super-block
    assert K % SUPER == 0 and group in GROUPS
    assert codes.shape == (P, N, K // group) and d_bits.shape == (N, J)
    total, off, payload, blk = packed_sizes(P, group, N, K)
    NT = -(-N // ROW_TILE)
    Np = NT * ROW_TILE
    beta = np.zeros((P, Np, K), dtype=np.uint32)
    beta[:, :N] = np.unpackbits(bits, axis=-1, bitorder="little")
    # beta[p][t*128 + r][256j + 128h + 32w + 2i + o] -> axes [p][t][r][j][h][w][i][o]
    b8 = beta.reshape(P, NT, ROW_TILE, J, 2, 4, 16, 2)
    shift = (np.arange(16, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])          # [i][o]
    words = np.bitwise_or.reduce(np.bitwise_or.reduce(b8 << shift, axis=7), axis=6)  # [p][t][r][j][h][w]
    words = np.ascontiguousarray(words.transpose(1, 3, 0, 4, 2, 5)).astype("<u4")  # [t][j][p][h][r][w]
    a = np.zeros((P, Np, K // group), dtype=np.uint8)
    a[:, :N] = codes
    a = np.ascontiguousarray(a.reshape(P, NT, ROW_TILE, J, GJ).transpose(1, 3, 0, 4, 2))  # [t][j][p][g][r]
    d = np.zeros((Np, J), dtype=np.uint16)
    d[:N] = d_bits
    d = np.ascontiguousarray(d.reshape(NT, ROW_TILE, J).transpose(0, 2, 1)).astype("<u2")  # [t][j][r]
    sign_bytes, code_bytes = 4096 * P, 128 * P * GJ
    blocks = np.zeros((NT, J, blk), dtype=np.uint8)
    blocks[:, :, :sign_bytes] = words.reshape(NT, J, 1024 * P).view(np.uint8)
    blocks[:, :, sign_bytes:sign_bytes + code_bytes] = a.reshape(NT, J, code_bytes)
    blocks[:, :, sign_bytes + code_bytes:] = d.view(np.uint8).reshape(NT, J, 256)
    out = np.zeros(total, dtype=np.uint8)
    out[:HEADER_BYTES] = header_bytes(N, K, P, group, payload, blk)
    out[off:] = blocks.reshape(-1)
    return out


def unpack(packed: np.ndarray):
    """Packed bytes -> (sign bits uint8 [P][N][K/8], codes uint8 [P][N][K/G],
    fp16 d bits [N][K/256], G)."""
    hd = parse_header(packed)
    assert hd["magic"] == MAGIC and hd["format"] == FORMAT_SA and hd["version"] == VERSION
    P, N, K, group = hd["P"], hd["N"], hd["K"], hd["group"]
    J, GJ = K // SUPER, SUPER // group
    NT = -(-N // ROW_TILE)
    blk = block_bytes(P, group)
    blocks = np.ascontiguousarray(
        packed[hd["payload_offset"]:hd["payload_offset"] + hd["payload_bytes"]]).reshape(NT, J, blk)
    sign_bytes, code_bytes = 4096 * P, 128 * P * GJ
    words = np.ascontiguousarray(blocks[:, :, :sign_bytes]).view("<u4").reshape(NT, J, P, 2, ROW_TILE, 4)
    shift = (np.arange(16, dtype=np.uint32)[:, None]
             + 16 * np.arange(2, dtype=np.uint32)[None, :])
    b = (words[..., None, None] >> shift) & np.uint32(1)             # [t][j][p][h][r][w][i][o]
    b = b.transpose(2, 0, 4, 1, 3, 5, 6, 7).reshape(P, NT * ROW_TILE, K)[:, :N]
    bits = np.packbits(b.astype(np.uint8), axis=-1, bitorder="little")
    a = blocks[:, :, sign_bytes:sign_bytes + code_bytes].reshape(NT, J, P, GJ, ROW_TILE)
    codes = np.ascontiguousarray(a.transpose(2, 0, 4, 1, 3).reshape(P, NT * ROW_TILE, K // group)[:, :N])
    d = np.ascontiguousarray(blocks[:, :, sign_bytes + code_bytes:]).view("<u2").reshape(NT, J, ROW_TILE)
    d_bits = np.ascontiguousarray(d.transpose(0, 2, 1).reshape(NT * ROW_TILE, J)[:N]).astype(np.uint16)
    return bits, codes, d_bits, group
