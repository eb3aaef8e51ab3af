"""Seeded synthetic workloads for the low-bit weight GEMV/GEMM path.

This module only *draws inputs*: random INT4 codes and scales, binary sign planes and
their per-plane scales, bf16 activations and draft token ids.  It holds none of the
method's arithmetic (no dequantisation, no products, no argmax, no acceptance rule), so
both the CPU oracle and the CUDA path can consume the same bytes without sharing code.

Every value is drawn in fp64 from numpy's PCG64 and rounded once, to nearest-even, into
the storage type (fp16 for scales and plane scales, bf16 for activations).  The draw
order inside one problem is fixed: codes, scales, plane scales, sign bits, activations,
drafts.  A problem's generator is seeded from ``SeedSequence([seed, *sub])`` so every
projection, batch size and plane count of a workload has its own reproducible stream.

Workload shapes follow the pages' models:
  * Efficient-Qwen report, section 2.1 and 3.3: INT4 symmetric per-group weights with
    group 128, 16-token draft blocks, a 4B-class dense decoder (hidden 2560).
  * ShiftAddQwen README, "Method" and "Format": binary planes w = sum_p alpha_p b_p.
  * Small-vocabulary MTP study, abstract and section 3.3: a 248,320-row vocabulary
    head and a trimmed 32,768-row head.
"""
from __future__ import annotations

import numpy as np

GROUP = 128

# Layer shapes of the 4B-class decoder: (name, K, N) for W[N][K].
LAYER_4B = (
    ("q", 2560, 4096),
    ("k", 2560, 1024),
    ("v", 2560, 1024),
    ("o", 2560, 2560),
    ("gate", 2560, 9728),
    ("up", 2560, 9728),
    ("down", 9728, 2560),
)

# Binary-plane matrices (K, N) and plane counts.
BINPLANE_SHAPES = ((4096, 12288), (12288, 4096))
BINPLANE_PLANES = (3, 4)

# Vocabulary heads: full and trimmed rows, hidden size K.
HEAD_K = 4096
HEAD_ROWS = (248_320, 32_768)

VERIFY_BLOCK = 16  # tokens in one draft block (one anchor/bonus row + 15 drafts)
M_SWEEP = (1, 2, 4, 8, 16, 32)

WORKLOADS = {
    "tiny": dict(name="tiny INT4 GEMV", kind="int4", M=1, shapes=((512, 256),), seed=0),
    "decode": dict(name="decode W4A16 GEMV, 4B-class layer", kind="int4", M=1,
                   shapes=tuple((k, n) for _, k, n in LAYER_4B), seed=1),
    "verify": dict(name="speculative-verify skinny GEMM, 4B-class layer", kind="int4", M=16,
                   shapes=tuple((k, n) for _, k, n in LAYER_4B), seed=2, m_sweep=M_SWEEP),
    "binplane": dict(name="binary-plane GEMV/GEMM", kind="binplane", M=(1, 16),
                     shapes=BINPLANE_SHAPES, planes=BINPLANE_PLANES, seed=3),
    "lmhead": dict(name="LM-head verify", kind="lmhead", M=VERIFY_BLOCK, K=HEAD_K,
                   rows=HEAD_ROWS, seed=4),
}


def generator(seed: int, *sub: int) -> np.random.Generator:
    """Independent PCG64 stream for (seed, sub...)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, sub)])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (round to nearest, ties to even); return uint16 bits.

    Works on the fp64 bit pattern: bf16 keeps 8 significant bits, so 45 of fp64's 52
    fraction bits are rounded away.  Inputs must be finite and inside bf16's normal
    range (true for every drawn activation).
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    b = x.view(np.uint64).copy()
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    r = b.view(np.float64)
    if not np.all(np.isfinite(r)):
        raise ValueError("activation out of bf16 range")
    # r is exactly representable in fp32 with the low 16 bits zero.
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to IEEE fp16 (numpy's conversion is round-to-nearest-even)."""
    h = np.asarray(x, dtype=np.float64).astype(np.float16)
    if not np.all(np.isfinite(h)):
        raise ValueError("value out of fp16 range")
    return h.view(np.uint16)


def int4_weights(g: np.random.Generator, N: int, K: int):
    """INT4 codes q ~ U{-8..7} (int8 [N][K]) and fp16 scales ~ LogNormal(ln 0.02, 0.3)
    (uint16 bits [N][K/128]); draw order: codes, then scales."""
    codes = g.integers(-8, 8, size=(N, K), dtype=np.int8)
    scales = to_f16_bits(g.lognormal(mean=np.log(0.02), sigma=0.3, size=(N, K // GROUP)))
    return codes, scales


def binplane_weights(g: np.random.Generator, P: int, N: int, K: int):
    """Binary planes: plane scales alpha [P][N][K/128] (fp16 bits) with
    alpha_1 ~ |N(0, 0.02)| and alpha_{p+1} = alpha_p * U(0.3, 0.6) chained in fp64 from
    the unrounded alpha_p, each rounded to fp16 at the end; then sign bits
    uint8 [P][N][K/8] with each bit uniform (bit j of byte b is element 8b+j, 1 means +1)."""
    G = K // GROUP
    a = np.empty((P, N, G), dtype=np.float64)
    a[0] = np.abs(g.normal(0.0, 0.02, size=(N, G)))
    for p in range(1, P):
        a[p] = a[p - 1] * g.uniform(0.3, 0.6, size=(N, G))
    alpha = to_f16_bits(a)
    bits = g.integers(0, 256, size=(P, N, K // 8), dtype=np.uint8)
    return bits, alpha


def activations(g: np.random.Generator, M: int, K: int) -> np.ndarray:
    """bf16 activation rows X[M][K] ~ N(0, 1), as uint16 bits."""
    return to_bf16_bits(g.standard_normal(size=(M, K)))


# The deployed ShiftAdd format (ShiftAddQwen README, "Format"): Q sign planes per super-block
# of 256 inputs, a u8 scale code per plane and group of G inputs, one fp16 d per super-block.
SA_GROUPS = (64, 128, 256)
SA_SHAPES = BINPLANE_SHAPES
SA_TYPES = ((3, 64), (4, 128))   # (planes, group) of the benchmark rows: sa3 and sa4_128


def sa_weights(g: np.random.Generator, P: int, N: int, K: int, G: int):
    """sa-format weights: d fp16 bits [N][K/256] ~ |N(0, 0.02)| / 255; codes uint8
    [P][N][K/G] with a_1 ~ U{128..255} and a_{p+1} = max(1, round(a_p * U(0.3, 0.6))) (the
    plane-scale decay of the binary-plane workload on the u8 grid); sign bits uint8
    [P][N][K/8] uniform.  Draw order: d, codes, bits."""
    d = to_f16_bits(np.abs(g.normal(0.0, 0.02, size=(N, K // 256))) / 255.0)
    a = np.empty((P, N, K // G), dtype=np.float64)
    a[0] = g.integers(128, 256, size=(N, K // G))
    for p in range(1, P):
        a[p] = np.maximum(1.0, np.rint(a[p - 1] * g.uniform(0.3, 0.6, size=(N, K // G))))
    codes = a.astype(np.uint8)
    bits = g.integers(0, 256, size=(P, N, K // 8), dtype=np.uint8)
    return bits, codes, d


def sa_problem(seed: int, P: int, G: int, M: int, N: int, K: int, *sub: int):
    """One sa-format problem: (bits, codes, d, X)."""
    g = generator(seed, 0x5A, P, G, M, N, K, *sub)
    bits, codes, d = sa_weights(g, P, N, K, G)
    x = activations(g, M, K)
    return bits, codes, d, x


# The trimmed draft head (Small-vocabulary MTP study, section 3.3): the 32,768 most used rows of
# the 248,320-row vocabulary, in NVFP4.
DRAFT_ROWS = HEAD_ROWS[1]


def nvfp4_weights(g: np.random.Generator, N: int, K: int):
    """NVFP4 weights: codes uint8 [N][K/2] (two 4-bit E2M1 codes per byte, each uniform over
    the 16 codes), E4M3 scale bytes uint8 [N][K/16] with exponent field uniform in 4..8 and
    mantissa uniform (normal values 2^-3 .. 3.75), tensor scale 0.01.  Draw order: codes,
    scales."""
    codes = g.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    e = g.integers(4, 9, size=(N, K // 16))
    m = g.integers(0, 8, size=(N, K // 16))
    scales = ((e << 3) | m).astype(np.uint8)
    return codes, scales, 0.01


def id_map(g: np.random.Generator, rows: int, vocab: int = HEAD_ROWS[0]) -> np.ndarray:
    """int32 [rows]: distinct full-vocabulary ids for the rows of a trimmed head."""
    return np.sort(g.choice(vocab, size=rows, replace=False)).astype(np.int32)


def nvfp4_problem(seed: int, M: int, N: int, K: int, *sub: int):
    """One draft-head problem: (codes, scales, g, id_map, H)."""
    gen = generator(seed, 0xF4, M, N, K, *sub)
    codes, scales, gs = nvfp4_weights(gen, N, K)
    ids = id_map(gen, N)
    h = activations(gen, M, K)
    return codes, scales, gs, ids, h


def q8_weights(g: np.random.Generator, N: int, K: int):
    """Q8 weights (the study's 8-bit head): codes int8 [N][K] uniform in [-127, 127] (the range
    a symmetric 8-bit quantiser rounds onto), fp16 scales [N][K/32] ~ LogNormal(ln(0.02/64),
    0.3), so weights are of order 0.02.  Draw order: codes, scales."""
    codes = g.integers(-127, 128, size=(N, K), dtype=np.int64).astype(np.int8)
    scales = to_f16_bits(g.lognormal(np.log(0.02 / 64), 0.3, size=(N, K // 32)))
    return codes, scales


def q8_problem(seed: int, M: int, N: int, K: int, *sub: int):
    """One Q8 draft-head problem: (codes, scales, id_map, H)."""
    gen = generator(seed, 0x08, M, N, K, *sub)
    codes, scales = q8_weights(gen, N, K)
    ids = id_map(gen, N)
    h = activations(gen, M, K)
    return codes, scales, ids, h


ACTIVATION_KINDS = ("outlier", "mixed_scale", "tiny", "huge", "zero", "sparse")


def activation_variant(g: np.random.Generator, M: int, K: int, kind: str) -> np.ndarray:
    """bf16 activation rows X[M][K] (uint16 bits) with a magnitude structure other than
    N(0, 1), drawn from one N(0, 1) matrix z and then, for each kind:
      outlier     -- each channel is, with probability 1/256, multiplied by 1000 in every row
                     (the few huge channels of decoder activations);
      mixed_scale -- each run of 64 inputs of a row multiplied by 2^e, e ~ U{-30..30};
      tiny / huge -- all of z times 2^-90 / 2^90;
      zero        -- all zero;
      sparse      -- each entry kept with probability 1/10, else zero (post-ReLU-like)."""
    z = g.standard_normal(size=(M, K))
    if kind == "outlier":
        z = z * np.where(g.random(K) < 1 / 256, 1000.0, 1.0)[None, :]
    elif kind == "mixed_scale":
        e = g.integers(-30, 31, size=(M, (K + 63) // 64))
        z = z * np.ldexp(1.0, np.repeat(e, 64, axis=1)[:, :K])
    elif kind == "tiny":
        z = np.ldexp(z, -90)
    elif kind == "huge":
        z = np.ldexp(z, 90)
    elif kind == "zero":
        z = np.zeros_like(z)
    elif kind == "sparse":
        z = np.where(g.random(size=(M, K)) < 0.1, z, 0.0)
    else:
        raise ValueError(kind)
    return to_bf16_bits(z)


def int4_problem(seed: int, M: int, N: int, K: int, *sub: int):
    """One INT4 problem: (codes, scales, X) drawn in that order."""
    g = generator(seed, M, N, K, *sub)
    codes, scales = int4_weights(g, N, K)
    x = activations(g, M, K)
    return codes, scales, x


def binplane_problem(seed: int, P: int, M: int, N: int, K: int, *sub: int):
    """One binary-plane problem: (bits, alpha, X) drawn as alpha, bits, X."""
    g = generator(seed, P, M, N, K, *sub)
    bits, alpha = binplane_weights(g, P, N, K)
    x = activations(g, M, K)
    return bits, alpha, x


def plant_drafts(seed: int, target_ids: np.ndarray, vocab: int, j: int | None = None):
    """Draft ids for a verify block of M = len(target_ids) rows.

    ``target_ids`` are the ids the target model is taken to predict at each row (the
    caller passes the oracle's argmax).  The first j drafts copy them, the rest are
    uniform over the vocabulary excluding the target's id at that row, so exactly j
    drafts are accepted.  j ~ U{0..M-1} unless given.  Returns (drafts int32 [M-1], j).
    """
    target_ids = np.asarray(target_ids, dtype=np.int64)
    M = target_ids.shape[0]
    g = generator(seed, 0xD2AF7, M, vocab)
    if j is None:
        j = int(g.integers(0, M))
    d = np.empty(M - 1, dtype=np.int32)
    for i in range(M - 1):
        if i < j:
            d[i] = target_ids[i]
        else:
            r = int(g.integers(0, vocab - 1))
            d[i] = r if r < target_ids[i] else r + 1
    return d, j
