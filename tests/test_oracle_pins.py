"""Pins for the CPU oracle: each check ties an oracle function to something other than
itself (hand-worked examples, brute force written another way, closed forms, invariants,
library rounding routines), so a dropped term, a wrong sign or index or a transposed
operand in the oracle fails here.  CPU only."""
import hashlib
import os

import numpy as np
import pytest
import torch

import synth
from oracle import q8, binplane, int4, numerics, nvfp4, sa, verify
from oracle.numerics import bf16_to_f64, f16_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                key, vals = line.split(":", 1)
                rows[key.strip()] = vals.split()
    return rows


def _bf16(vals):
    return numerics.bf16_bits(numerics.round_to_bf16(np.asarray(vals, dtype=np.float64)))


def _f16(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


# ------------------------------------------------------------------ numerics

def test_round_to_bf16_matches_torch_on_fp32_values():
    g = np.random.default_rng(11)
    x32 = np.concatenate([
        g.standard_normal(20000).astype(np.float32),
        (g.standard_normal(5000) * 1e-30).astype(np.float32),
        (g.standard_normal(5000) * 1e30).astype(np.float32),
        # exact ties between two bf16 neighbours: 1 + 2^-8, 1 + 3*2^-8, -(2 + 2^-7)
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(2 + 2 ** -7), 0.0, -0.0], dtype=np.float32),
    ])
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = numerics.bf16_bits(numerics.round_to_bf16(x32.astype(np.float64)))
    assert np.array_equal(got, ref)


def test_round_to_bf16_ties_by_hand():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even neighbour, 1.
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: even neighbour is 1 + 2^-6.
    # Just above a tie rounds up.
    r = numerics.round_to_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40,
                                         255.5, 256.5 * 2, -3.0]))
    assert list(r) == [1.0, 1 + 2 ** -6, 1 + 2 ** -7, 256.0, 512.0, -3.0]


def test_decoders_are_exact():
    v = np.array([0.5, -2.0, 1.0 / 3.0, 65504.0, 6.1e-5])
    assert np.array_equal(numerics.f16_to_f64(_f16(v)), v.astype(np.float16).astype(np.float64))
    x = np.array([1.0, -0.15625, 3.0e38, 1e-38])
    bits = _bf16(x)
    assert np.array_equal(numerics.bf16_to_f64(bits), numerics.round_to_bf16(x))


def test_generator_roundings_are_representable_and_deterministic():
    codes, scales, x = synth.int4_problem(0, 1, 256, 512)
    assert codes.min() >= -8 and codes.max() <= 7
    # drawn bf16 values are a fixed point of the oracle's rounding
    xv = numerics.bf16_to_f64(x)
    assert np.array_equal(numerics.round_to_bf16(xv), xv)
    h = hashlib.sha256(codes.tobytes() + scales.tobytes() + x.tobytes()).hexdigest()
    codes2, scales2, x2 = synth.int4_problem(0, 1, 256, 512)
    assert h == hashlib.sha256(codes2.tobytes() + scales2.tobytes() + x2.tobytes()).hexdigest()
    # the generator's own bf16 rounding agrees with the oracle's on fresh fp64 draws
    d = np.random.default_rng(5).standard_normal(50000)
    assert np.array_equal(synth.to_bf16_bits(d), _bf16(d))


# ------------------------------------------------------------------ INT4

@pytest.mark.parametrize("G", [4, 8])
def test_int4_hand_example(G):
    fx = _read_fixture("int4_hand_4x8.txt")
    x = _bf16([float(v) for v in fx["x"]])[None, :]
    q = np.array([[int(v) for v in fx[f"q{n}"]] for n in range(4)], dtype=np.int8)
    s = _f16([[float(v) for v in fx[f"G{G}_s{n}"]] for n in range(4)])
    y = int4.gemm(x, q, s, group=G)
    assert np.array_equal(y[0], np.array([float(v) for v in fx[f"G{G}_y"]]))


def _brute_int4(xv, q, s, G):
    # group-sum-first, pure Python loops: sum_g s * (sum_{k in g} q * x)
    M, K = xv.shape
    N = q.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for g in range(K // G):
                part = 0.0
                for k in range(g * G, (g + 1) * G):
                    part += int(q[n, k]) * float(xv[m, k])
                tot += float(s[n, g]) * part
            out[m, n] = tot
    return out


@pytest.mark.parametrize("M,N,K", [(1, 3, 128), (2, 5, 256), (3, 2, 384)])
def test_int4_brute_force(M, N, K):
    codes, scales, x = synth.int4_problem(123, M, N, K)
    y = int4.gemm(x, codes, scales)
    ref = _brute_int4(numerics.bf16_to_f64(x), codes, numerics.f16_to_f64(scales), 128)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_int4_one_hot_and_group_closed_forms():
    N, K = 7, 384
    codes, scales, _ = synth.int4_problem(9, 1, N, K)
    sv = numerics.f16_to_f64(scales)
    # one-hot activation at k picks column k of W: y = RNE(s[n][k//128] * q[n][k])
    for k in (0, 127, 128, 200, 383):
        x = np.zeros((1, K)); x[0, k] = 1.0
        y = int4.gemm(_bf16(x), codes, scales)
        assert np.array_equal(y[0], sv[:, k // 128] * codes[:, k])
    # x = 1 on one group: y = s * sum_{k in g} q
    x = np.zeros((1, K)); x[0, 128:256] = 1.0
    y = int4.gemm(_bf16(x), codes, scales)
    assert np.array_equal(y[0], sv[:, 1] * codes[:, 128:256].sum(axis=1))
    # zero scales give exact zeros
    y = int4.gemm(_bf16(np.ones((1, K))), codes, np.zeros_like(scales))
    assert np.all(y == 0)


def test_int4_layout_positions_by_hand():
    N, K = 200, 256
    rows = []
    with open(os.path.join(GOLDEN, "int4_layout_positions.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                n, k, byte, nib = line.split()
                rows.append((int(n), int(k), int(byte), nib))
    total, off, payload, block = int4.packed_sizes(N, K)
    assert (off, payload, block) == (128, 33792, 8448)
    code_bytes = np.zeros(payload, dtype=bool)      # which payload bytes hold codes
    for b in range(4):
        code_bytes[b * block:b * block + 8192] = True
    for n, k, byte, nib in rows:
        codes = np.zeros((N, K), dtype=np.int8)
        codes[n, k] = 5                              # nibble u = 13, every other nibble 8
        packed = int4.pack(codes, np.zeros((N, K // 128), dtype=np.uint16))
        sec = packed[off:off + payload]
        lo, hi = sec & 0xF, sec >> 4
        expect_lo = np.where(code_bytes, 8, 0); expect_hi = np.where(code_bytes, 8, 0)
        (expect_lo if nib == "lo" else expect_hi)[byte] = 13
        assert np.array_equal(lo, expect_lo) and np.array_equal(hi, expect_hi), (n, k)
    scales = np.zeros((N, K // 128), dtype=np.uint16)
    scales[130, 1] = 0x3C00
    packed = int4.pack(np.zeros((N, K), dtype=np.int8), scales)
    sec = packed[off:off + payload].copy()
    sec[code_bytes] = 0
    sec = sec.view("<u2")
    assert sec[33540 // 2] == 0x3C00 and np.count_nonzero(sec) == 1


@pytest.mark.parametrize("N,K", [(40, 256), (256, 512), (33, 128), (300, 384)])
def test_int4_pack_round_trip_and_header(N, K):
    codes, scales, _ = synth.int4_problem(4, 1, N, K)
    packed = int4.pack(codes, scales)
    assert packed.size == int4.packed_sizes(N, K)[0]
    c2, s2 = int4.unpack(packed)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    hd = int4.parse_header(packed)
    assert (hd["magic"], hd["format"], hd["N"], hd["K"], hd["group"]) == (int4.MAGIC, 1, N, K, 128)
    # exactly N*K/2 + N*K/64 payload bytes when N is a multiple of the 128-row tile
    if N % 128 == 0:
        assert hd["payload_bytes"] == N * K // 2 + N * K // 64


# ------------------------------------------------------------------ binary planes

@pytest.mark.parametrize("G", [4, 8])
def test_binplane_hand_example(G):
    fx = _read_fixture("binplane_hand_4x8.txt")
    x = _bf16([float(v) for v in fx["x"]])[None, :]
    bits = np.array([[[int(v, 16)] for v in fx["bits_p0"]],
                     [[int(v, 16)] for v in fx["bits_p1"]]], dtype=np.uint8)   # [2][4][1]
    a0 = np.array([float(v) for v in fx[f"G{G}_a_p0"]]).reshape(4, -1)
    a1 = np.array([float(v) for v in fx[f"G{G}_a_p1"]]).reshape(4, -1)
    alpha = _f16(np.stack([a0, a1]))
    y = binplane.gemm(x, bits, alpha, group=G)
    assert np.array_equal(y[0], np.array([float(v) for v in fx[f"G{G}_y"]]))


def test_binplane_planes_are_exactly_pm1_and_identity():
    bits, alpha, x = synth.binplane_problem(3, 3, 1, 8, 256)
    b = binplane.signs(bits)
    assert set(np.unique(b)) == {-1.0, 1.0}
    # sum b*x = 2 * sum_{b=+1} x - sum x, on random data
    xv = numerics.bf16_to_f64(x)[0]
    lhs = b @ xv
    rhs = 2 * ((b > 0) * xv).sum(axis=-1) - xv.sum()
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


def test_binplane_closed_forms():
    P, N, K = 1, 5, 256
    _, alpha, x = synth.binplane_problem(8, P, 1, N, K)
    xv = numerics.bf16_to_f64(x)[0]
    av = numerics.f16_to_f64(alpha)[0]
    gsum = xv.reshape(2, 128).sum(axis=1)
    ones = np.full((P, N, K // 8), 0xFF, dtype=np.uint8)
    zeros = np.zeros((P, N, K // 8), dtype=np.uint8)
    assert np.allclose(binplane.gemm(x, ones, alpha)[0], av @ gsum, rtol=1e-14, atol=0)
    assert np.allclose(binplane.gemm(x, zeros, alpha)[0], -(av @ gsum), rtol=1e-14, atol=0)
    # one-hot activation picks sum_p alpha_p b_p at that input
    bits, alpha, _ = synth.binplane_problem(8, 4, 1, N, K)
    for k in (0, 7, 8, 129, 255):
        xo = np.zeros((1, K)); xo[0, k] = 1.0
        y = binplane.gemm(_bf16(xo), bits, alpha)[0]
        sgn = ((bits[:, :, k // 8] >> (k % 8)) & 1) * 2.0 - 1.0     # [P][N]
        assert np.array_equal(y, (numerics.f16_to_f64(alpha)[:, :, k // 128] * sgn).sum(axis=0))


def test_binplane_brute_force():
    P, M, N, K = 3, 2, 3, 256
    bits, alpha, x = synth.binplane_problem(21, P, M, N, K)
    xv = numerics.bf16_to_f64(x)
    av = numerics.f16_to_f64(alpha)
    ref = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            tot = 0.0
            for p in range(P):
                for g in range(K // 128):
                    s = 0.0
                    for k in range(g * 128, (g + 1) * 128):
                        bit = (int(bits[p, n, k // 8]) >> (k % 8)) & 1
                        s += xv[m, k] if bit else -xv[m, k]
                    tot += av[p, n, g] * s
            ref[m, n] = tot
    assert np.allclose(binplane.gemm(x, bits, alpha), ref, rtol=1e-12, atol=1e-14)


def test_binplane_layout_positions_by_hand():
    P, N, K = 2, 200, 256
    total, off, payload, block = binplane.packed_sizes(P, N, K)
    assert block == 4608
    with open(os.path.join(GOLDEN, "binplane_layout_positions.txt")) as f:
        rows = [tuple(int(v) for v in line.split()) for line in f
                if line.strip() and not line.startswith("#")]
    for p, n, k, byte, bit in rows:
        bits = np.zeros((P, N, K // 8), dtype=np.uint8)
        bits[p, n, k // 8] = 1 << (k % 8)
        packed = binplane.pack(bits, np.zeros((P, N, K // 128), dtype=np.uint16))
        sec = packed[off:off + payload]
        expect = np.zeros(payload, dtype=np.uint8)
        expect[byte] = 1 << bit
        assert np.array_equal(sec, expect), (p, n, k)


@pytest.mark.parametrize("P,N,K", [(2, 40, 256), (3, 128, 512), (4, 33, 128), (1, 256, 256)])
def test_binplane_pack_round_trip(P, N, K):
    bits, alpha, _ = synth.binplane_problem(6, P, 1, N, K)
    packed = binplane.pack(bits, alpha)
    b2, a2 = binplane.unpack(packed)
    assert np.array_equal(b2, bits) and np.array_equal(a2, alpha)
    if N % 128 == 0:
        hd = int4.parse_header(packed)
        assert hd["payload_bytes"] == P * N * K // 8 + P * N * K // 64


# ------------------------------------------------------------------ argmax / acceptance

def test_argmax_lowest_index_brute_force():
    g = np.random.default_rng(3)
    for _ in range(200):
        L = g.integers(-3, 4, size=(3, 9)).astype(np.float64)   # many ties
        a = verify.argmax_lowest(L)
        for r in range(3):
            best = max(L[r])
            assert a[r] == min(i for i in range(9) if L[r, i] == best)


def test_argmax_planted_maximum():
    N, K = 300, 256
    codes, scales, x = synth.int4_problem(17, 2, N, K)
    # row 123 = +7 where x > 0 and -8 where x <= 0 with a large scale: it dominates every row
    xv = numerics.bf16_to_f64(x)
    codes[123] = np.where(xv[0] > 0, 7, -8)
    scales[123] = _f16(np.full(K // 128, 4.0))
    a = verify.argmax_lowest(int4.gemm(x, codes, scales))
    assert a[0] == 123


def test_top2_margin():
    L = np.array([[1.0, 3.0, 2.5], [4.0, 4.0, 0.0]])
    assert np.array_equal(verify.top2_margin(L), [0.5, 0.0])


def test_acceptance_exhaustive_small_alphabet():
    # every (a, d) over a 3-letter alphabet with M = 4 rows: compare with a direct count
    import itertools
    for a in itertools.product(range(3), repeat=4):
        for d in itertools.product(range(3), repeat=3):
            n, bonus = verify.accept(a, d)
            k = 0
            for i in range(3):
                if all(d[j] == a[j] for j in range(i + 1)):
                    k = i + 1
            assert n == k and bonus == a[k] and 1 <= n + 1 <= 4


def test_acceptance_planted_drafts():
    a = np.arange(16) * 7 + 3
    for j in range(16):
        d, jj = synth.plant_drafts(5, a, 1000, j=j)
        assert jj == j
        n, bonus = verify.accept(a, d)
        assert n == j and bonus == a[j]
    d, j = synth.plant_drafts(5, a, 1000)
    assert verify.accept(a, d)[0] == j


# ----------------------------------------------------------------------------- sa format
# ShiftAddQwen README, "Format": per super-block of 256 inputs, Q sign planes, a u8 code per
# plane and group of G inputs, one fp16 d; alpha = d * a.

def _sa_hand_inputs():
    P, N, K = 2, 2, 256
    x = np.zeros((1, K))
    x[0, :4] = [1, 2, 3, 4]
    x[0, 128], x[0, 255] = 5, -1
    bits = np.zeros((P, N, K // 8), dtype=np.uint8)
    bits[0, 0, 0], bits[0, 0, 16], bits[0, 0, 31] = 0x05, 0x01, 0x80
    bits[1, 0, 0] = 0x0F
    bits[:, 1, :] = 0xFF
    d = synth.to_f16_bits(np.array([[0.5], [0.25]]))
    return synth.to_bf16_bits(x), bits, d


def test_sa_hand_example():
    x, bits, d = _sa_hand_inputs()
    with open(os.path.join(GOLDEN, "sa_hand_2x256.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    assert len(rows) == 3
    for G, c0, c1, y0, y1 in rows:
        G = int(G)
        a0 = [int(v) for v in c0.split(",")]
        a1 = [int(v) for v in c1.split(",")]
        codes = np.zeros((2, 2, 256 // G), dtype=np.uint8)
        codes[0, :, :] = a0
        codes[1, :, :] = a1
        Y = sa.gemm(x, bits, codes, d, G)
        assert Y[0, 0] == float(y0) and Y[0, 1] == float(y1), (G, Y)


@pytest.mark.parametrize("G", sa.GROUPS)
def test_sa_equals_fp16_alpha_planes_when_exact(G):
    """With G = 128 and d * a exact in fp16, the sa weights are the fp16-alpha binary planes
    with alpha = d * a; for G = 64 / 256 the same holds after expanding alpha to groups of 128
    (G = 64: the two halves share one alpha only when their codes agree, so they are set equal)."""
    P, N, K = 3, 40, 512
    g = synth.generator(11, P, N, K, G)
    bits = g.integers(0, 256, size=(P, N, K // 8), dtype=np.uint8)
    codes = g.integers(1, 256, size=(P, N, K // G), dtype=np.uint8)
    if G == 64:
        codes[..., 1::2] = codes[..., 0::2]
    d = synth.to_f16_bits(np.ldexp(g.integers(1, 8, size=(N, K // 256)).astype(float), -12))
    x = synth.activations(g, 2, K)
    dd = np.repeat(f16_to_f64(d), 2, axis=1)                                  # per group of 128
    a128 = codes.astype(float)[..., ::2] if G == 64 else (
        np.repeat(codes.astype(float), 2, axis=2) if G == 256 else codes.astype(float))
    alpha = synth.to_f16_bits(dd[None] * a128)
    assert np.array_equal(f16_to_f64(alpha), dd[None] * a128)               # exact in fp16
    assert np.array_equal(sa.gemm(x, bits, codes, d, G), binplane.gemm(x, bits, alpha))


@pytest.mark.parametrize("G", sa.GROUPS)
def test_sa_brute_force(G):
    P, N, K = 2, 3, 512
    bits, codes, d, x = synth.sa_problem(12, P, G, 2, N, K)
    X = bf16_to_f64(x)
    dv = f16_to_f64(d)
    ref = np.zeros((2, N))
    for m in range(2):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                w = 0.0
                for p in range(P):
                    sgn = 1.0 if (bits[p, n, k // 8] >> (k % 8)) & 1 else -1.0
                    w += float(codes[p, n, k // G]) * sgn
                acc += X[m, k] * dv[n, k // 256] * w
            ref[m, n] = acc
    Y = sa.gemm(x, bits, codes, d, G)
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
    # the sampled-rows form used on full-size matrices: the same brute-force values, per row
    for rows in ([2], [0, 2], [2, 0, 1]):
        assert np.allclose(sa.gemm_entries(x, bits, codes, d, G, np.array(rows)), ref[:, rows],
                           rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("G", sa.GROUPS)
def test_sa_group_and_superblock_locality(G):
    """Only group g's code nonzero: the output depends on inputs of group g alone and scales
    with that super-block's d; all signs +1 gives the closed form d * a * sum of the group."""
    P, N, K = 2, 5, 768
    g = synth.generator(13, G)
    bits = np.full((P, N, K // 8), 0xFF, dtype=np.uint8)
    d = synth.to_f16_bits(g.uniform(0.5, 2.0, size=(N, K // 256)))
    x = synth.activations(g, 1, K)
    X = bf16_to_f64(x)[0]
    for grp in (0, K // G - 1, (K // G) // 2):
        codes = np.zeros((P, N, K // G), dtype=np.uint8)
        codes[0, :, grp], codes[1, :, grp] = 3, 5
        Y = sa.gemm(x, bits, codes, d, G)[0]
        ks = slice(grp * G, (grp + 1) * G)
        expect = f16_to_f64(d)[:, (grp * G) // 256] * 8.0 * X[ks].sum()
        assert np.allclose(Y, expect, rtol=1e-13, atol=0)
        x2 = x.copy()
        x2[0, ks] = 0
        assert not np.any(sa.gemm(x2, bits, codes, d, G))


def test_sa_layout_positions_by_hand():
    P, N, K, G = 2, 200, 512, 64
    total, off, payload, block = sa.packed_sizes(P, G, N, K)
    assert block == 9472 and payload == 2 * 2 * 9472
    with open(os.path.join(GOLDEN, "sa_layout_positions.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    zb = np.zeros((P, N, K // 8), dtype=np.uint8)
    zc = np.zeros((P, N, K // G), dtype=np.uint8)
    zd = np.zeros((N, K // 256), dtype=np.uint16)
    for kind, p, n, kg, byte, bit in rows:
        n, kg, byte = int(n), int(kg), int(byte)
        bits, codes, d = zb.copy(), zc.copy(), zd.copy()
        expect = np.zeros(payload, dtype=np.uint8)
        if kind == "sign":
            bits[int(p), n, kg // 8] = 1 << (kg % 8)
            expect[byte] = 1 << int(bit)
        elif kind == "code":
            codes[int(p), n, kg] = 0xA5
            expect[byte] = 0xA5
        else:
            d[n, kg] = 0x3C01
            expect[byte], expect[byte + 1] = 0x01, 0x3C
        sec = sa.pack(bits, codes, d, G)[off:off + payload]
        assert np.array_equal(sec, expect), (kind, p, n, kg)


@pytest.mark.parametrize("P,G,N,K", [(2, 64, 40, 256), (3, 128, 128, 512), (6, 64, 33, 256),
                                     (1, 256, 256, 768), (4, 128, 129, 1024)])
def test_sa_pack_round_trip(P, G, N, K):
    bits, codes, d, _ = synth.sa_problem(14, P, G, 1, N, K)
    packed = sa.pack(bits, codes, d, G)
    b2, c2, d2, g2 = sa.unpack(packed)
    assert g2 == G and np.array_equal(b2, bits) and np.array_equal(c2, codes) and np.array_equal(d2, d)
    hd = int4.parse_header(packed)
    assert hd["format"] == sa.FORMAT_SA and hd["group"] == G and hd["P"] == P
    if N % 128 == 0:   # payload = sign bits + u8 codes + fp16 d, nothing else
        assert hd["payload_bytes"] == P * N * K // 8 + P * N * K // G + 2 * N * K // 256


# ----------------------------------------------------------------------------- NVFP4 head
# Small-vocabulary MTP study, section 3.3: the trimmed draft head in NVFP4 (E2M1 weights, an
# E4M3 scale per 16, an fp32 tensor scale), draft ids mapped to the full vocabulary.

def test_e2m1_values_are_the_published_list():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(nvfp4.e2m1_to_f64(np.arange(8))) == mags
    assert list(nvfp4.e2m1_to_f64(np.arange(8, 16))) == [-m for m in mags]


def test_e4m3_decode_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = nvfp4.e4m3_to_f64(b)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_nvfp4_hand_example():
    rows = _read_fixture("nvfp4_hand_1x32.txt")
    K = 32
    codes = np.zeros((1, K // 2), dtype=np.uint8)
    for kv in rows["codes"]:
        i, v = kv.split(":")
        codes[0, int(i)] = int(v, 16)
    scales = np.array([[int(v, 16) for v in rows["scales"]]], dtype=np.uint8)
    x = np.zeros((1, K))
    for kv in rows["x"]:
        i, v = kv.split(":")
        x[0, int(i)] = float(v)
    y = nvfp4.gemm(synth.to_bf16_bits(x), codes, scales, float(rows["g"][0]))
    assert y[0, 0] == float(rows["y"][0])


def test_nvfp4_brute_force():
    codes, scales, g, _, h = synth.nvfp4_problem(30, 2, 5, 128)
    H = numerics.bf16_to_f64(h)
    ref = np.zeros((2, 5))
    for m in range(2):
        for n in range(5):
            acc = 0.0
            for k in range(128):
                c = (codes[n, k // 2] >> (4 * (k % 2))) & 15
                sgn = -1.0 if c & 8 else 1.0
                e, mm = (c >> 1) & 3, c & 1
                v = sgn * (mm * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + mm / 2))
                sb = int(scales[n, k // 16])
                se, sm = (sb >> 3) & 15, sb & 7
                sv = (sm / 8.0) * 2.0 ** -6 if se == 0 else 2.0 ** (se - 7) * (1 + sm / 8)
                acc += H[m, k] * np.float32(g) * sv * v
            ref[m, n] = acc
    assert np.allclose(nvfp4.gemm(h, codes, scales, g), ref, rtol=1e-12, atol=1e-12)


def test_nvfp4_layout_positions_by_hand():
    N, K = 200, 256
    total, off, payload, block = nvfp4.packed_sizes(N, K)
    assert block == 9216 and payload == 2 * 2 * 9216
    with open(os.path.join(GOLDEN, "nvfp4_layout_positions.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    for kind, n, kj, byte, nib in rows:
        n, kj, byte = int(n), int(kj), int(byte)
        codes = np.zeros((N, K // 2), dtype=np.uint8)
        scales = np.zeros((N, K // 16), dtype=np.uint8)
        expect = np.zeros(payload, dtype=np.uint8)
        if kind == "code":
            codes[n, kj // 2] = 0x5 << (4 * (kj % 2))
            expect[byte] = 0x5 << (4 * int(nib))
        else:
            scales[n, kj] = 0x3A
            expect[byte] = 0x3A
        sec = nvfp4.pack(codes, scales, 1.0)[off:off + payload]
        assert np.array_equal(sec, expect), (kind, n, kj)


@pytest.mark.parametrize("N,K", [(1, 128), (130, 256), (256, 512)])
def test_nvfp4_pack_round_trip(N, K):
    codes, scales, g, _, _ = synth.nvfp4_problem(31, 1, N, K)
    packed = nvfp4.pack(codes, scales, g)
    c2, s2, g2 = nvfp4.unpack(packed)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales) and g2 == np.float32(g)
    hd = int4.parse_header(packed)
    assert hd["format"] == nvfp4.FORMAT_NVFP4 and hd["block_bytes"] == 9216
    if N % 128 == 0:
        assert hd["payload_bytes"] == N * K // 2 + N * K // 16


def test_draft_ids_map_and_ties():
    logits = np.array([[1.0, 3.0, 3.0, -2.0], [0.0, -1.0, -5.0, 0.0]])
    ids = np.array([70, 11, 4, 9], dtype=np.int32)
    assert list(nvfp4.draft_ids(logits)) == [1, 0]          # lowest row among equal maxima
    assert list(nvfp4.draft_ids(logits, ids)) == [11, 70]
    g = synth.generator(32)
    L = g.standard_normal((5, 1000))
    m = synth.id_map(g, 1000)
    assert len(set(m.tolist())) == 1000
    assert np.array_equal(nvfp4.draft_ids(L, m), m[np.argmax(L, axis=1)])



# ------------------------------------------------------------------ Q8 (the 8-bit draft head)

def test_q8_hand_example():
    fx = _read_fixture("q8_hand_2x64.txt")
    K = 64
    codes = np.zeros((2, K), dtype=np.int8)
    codes[0, :32], codes[0, 32:] = 1, -2
    codes[0, 40] = -128
    codes[1] = (np.arange(K) % 4) - 1
    codes[1, 1] = 127
    d = _f16([[float(v) for v in fx["d0"]], [float(v) for v in fx["d1"]]])
    x = np.zeros((1, K))
    x[0, :48] = 1.0
    y = q8.gemm(_bf16(x), codes, d)
    assert np.array_equal(y[0], np.array([float(v) for v in fx["y"]]))


def test_q8_brute_force_and_closed_forms():
    codes, scales, _, h = synth.q8_problem(60, 2, 5, 256)
    H, dv = numerics.bf16_to_f64(h), numerics.f16_to_f64(scales)
    ref = np.zeros((2, 5))
    for m in range(2):
        for n in range(5):
            acc = 0.0
            for blk in range(256 // 32):  # block-sum-first, pure Python
                part = 0
                for k in range(32 * blk, 32 * blk + 32):
                    part += int(codes[n, k]) * float(H[m, k])
                acc += float(dv[n, blk]) * part
            ref[m, n] = acc
    assert np.allclose(q8.gemm(h, codes, scales), ref, rtol=1e-12, atol=1e-12)
    # one-hot activation picks d * q exactly; the extreme codes -128 and 127 decode as integers
    codes[0, 7], codes[1, 200] = -128, 127
    for n, k in ((0, 7), (1, 200), (4, 255)):
        x = np.zeros((1, 256)); x[0, k] = 1.0
        assert q8.gemm(_bf16(x), codes, scales)[0, n] == dv[n, k // 32] * int(codes[n, k])


def test_q8_layout_positions_by_hand():
    N, K = 200, 256
    total, off, payload, block = q8.packed_sizes(N, K)
    assert block == 17408 and payload == 2 * 2 * 17408
    with open(os.path.join(GOLDEN, "q8_layout_positions.txt")) as f:
        rows = [line.split() for line in f if line.strip() and not line.startswith("#")]
    for kind, n, kj, byte in rows:
        n, kj, byte = int(n), int(kj), int(byte)
        codes = np.zeros((N, K), dtype=np.int8)
        scales = np.zeros((N, K // 32), dtype=np.uint16)
        expect = np.zeros(payload, dtype=np.uint8)
        if kind == "code":
            codes[n, kj] = -3
            expect[byte] = 0xFD
        else:
            scales[n, kj] = 0x3C01
            expect[byte], expect[byte + 1] = 0x01, 0x3C
        assert np.array_equal(q8.pack(codes, scales)[off:off + payload], expect), (kind, n, kj)


@pytest.mark.parametrize("N,K", [(1, 128), (130, 256), (256, 512)])
def test_q8_pack_round_trip(N, K):
    codes, scales, _, _ = synth.q8_problem(61, 1, N, K)
    packed = q8.pack(codes, scales)
    c2, s2 = q8.unpack(packed)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    hd = int4.parse_header(packed)
    assert hd["format"] == q8.FORMAT_Q8 and hd["block_bytes"] == 17408
    if N % 128 == 0:
        assert hd["payload_bytes"] == N * K + N * (K // 32) * 2
