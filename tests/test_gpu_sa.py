"""GPU parity for the deployed ShiftAdd format (ShiftAddQwen README, "Format": u8 scale codes
per plane and group of G inputs, one fp16 d per 256 inputs, alpha = d * a) through the C ABI
against the CPU oracle (``oracle.sa``).  Inputs come from ``synth``; expected values only from
the oracle."""
import numpy as np
import pytest

import synth
from oracle import sa as osa
from helpers import bf16_dev, check_gemm, dev, f16_dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def pack_sa_gpu(lb, bits, codes, d, G):
    P, N, KB = bits.shape
    K = KB * 8
    packed = torch.empty(lb.lowbit_sa_packed_bytes(P, G, N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_sa(dev(bits), dev(codes), f16_dev(d), P, G, N, K, packed)
    return packed


def gemm_sa_gpu(lb, x, packed, P, G, M, N, K, path=0):
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_sa_path(bf16_dev(x), packed, P, G, M, N, K, Y, path)
    torch.cuda.synchronize()
    return host_bits(Y)


@pytest.mark.parametrize("P,G,N,K", [(2, 64, 40, 256), (3, 128, 128, 512), (6, 64, 33, 256),
                                     (1, 256, 257, 768), (4, 128, 129, 1024), (8, 64, 300, 512),
                                     (3, 64, 12288, 4096)])
def test_pack_sa_bit_exact(lb, P, G, N, K):
    bits, codes, d, _ = synth.sa_problem(20, P, G, 1, N, K)
    got = pack_sa_gpu(lb, bits, codes, d, G).cpu().numpy()
    ref = osa.pack(bits, codes, d, G)
    assert got.shape == ref.shape and np.array_equal(got, ref)
    b2, c2, d2, g2 = osa.unpack(got)
    assert g2 == G and np.array_equal(b2, bits) and np.array_equal(c2, codes) and np.array_equal(d2, d)


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("M", [1, 2, 3, 16, 32])
@pytest.mark.parametrize("P,G,N,K", [(1, 64, 1, 256), (2, 64, 65, 512), (3, 128, 257, 1280),
                                     (4, 256, 300, 768), (6, 64, 130, 256), (8, 128, 100, 512),
                                     (8, 64, 129, 512), (3, 256, 2000, 2048)])
def test_sa_small_and_ragged(lb, P, G, N, K, M, path):
    bits, codes, d, x = synth.sa_problem(21, P, G, M, N, K)
    y = gemm_sa_gpu(lb, x, pack_sa_gpu(lb, bits, codes, d, G), P, G, M, N, K, path)
    check_gemm(y, osa.gemm(x, bits, codes, d, G), f"sa P={P} G={G} M={M} N={N} K={K} path={path}")


@pytest.mark.parametrize("M,path", [(1, 0), (16, 0), (16, 1), (16, 2)])
@pytest.mark.parametrize("P,G", synth.SA_TYPES)
@pytest.mark.parametrize("shape", range(len(synth.SA_SHAPES)))
def test_sa_binary_plane_matrices(lb, shape, P, G, M, path):
    """The binary-plane workload's matrices (K, N) in {(4096, 12288), (12288, 4096)} in
    the deployed format; every output at M = 1, every output of 1024 sampled rows at M = 16."""
    K, N = synth.SA_SHAPES[shape]
    bits, codes, d, x = synth.sa_problem(3, P, G, M, N, K, shape)
    y = gemm_sa_gpu(lb, x, pack_sa_gpu(lb, bits, codes, d, G), P, G, M, N, K, path)
    if M == 1:
        check_gemm(y, osa.gemm(x, bits, codes, d, G), f"sa binary-plane shape {shape} M=1")
    else:
        rows = np.sort(synth.generator(22, shape).choice(N, size=1024, replace=False))
        check_gemm(y[:, rows], osa.gemm_entries(x, bits, codes, d, G, rows),
                   f"sa binary-plane shape {shape} M=16 sampled")


@pytest.mark.parametrize("M,path", [(1, 0), (16, 2), (16, 3)])
@pytest.mark.parametrize("kind", ("outlier", "mixed_scale", "tiny", "sparse"))
def test_sa_activation_structures(lb, kind, M, path):
    P, G, N, K = 3, 64, 260, 1024
    g = synth.generator(23, synth.ACTIVATION_KINDS.index(kind))
    bits, codes, d = synth.sa_weights(g, P, N, K, G)
    x = synth.activation_variant(g, M, K, kind)
    y = gemm_sa_gpu(lb, x, pack_sa_gpu(lb, bits, codes, d, G), P, G, M, N, K, path)
    check_gemm(y, osa.gemm(x, bits, codes, d, G), f"sa {kind} M={M} path={path}",
               scale=2.0 ** 90 if kind == "tiny" else 1.0)


@pytest.mark.parametrize("M,path", [(1, 0), (4, 1), (4, 2), (4, 3)])
@pytest.mark.parametrize("wrong", ["G", "P", "N"])
def test_sa_header_mismatch_leaves_outputs(lb, wrong, M, path):
    """A buffer packed for other (P, G, N) is rejected on the device: the error word is set and
    no output is written."""
    P, G, N, K = 3, 128, 200, 512
    bits, codes, d, x = synth.sa_problem(24, P, G, M, N, K)
    packed = pack_sa_gpu(lb, bits, codes, d, G)
    lb.lowbit_device_error()
    P2, G2, N2 = (P, 64 if wrong == "G" else G, N) if wrong != "P" else (2, G, N)
    if wrong == "N":
        N2 = N - 128
    Y = torch.full((M, N2), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_sa_path(bf16_dev(x), packed, P2, G2, M, N2, K, Y, path)
    assert lb.lowbit_device_error() == 1
    assert bool((Y == 7.0).all())


def test_sa_validation(lb):
    P, G, N, K = 2, 64, 64, 256
    bits, codes, d, x = synth.sa_problem(25, P, G, 1, N, K)
    packed = pack_sa_gpu(lb, bits, codes, d, G)
    X = torch.zeros((33, 512), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((33, N), dtype=torch.bfloat16, device="cuda")
    assert lb.lowbit_sa_packed_bytes(P, 32, N, K) == 0
    assert lb.lowbit_sa_packed_bytes(P, G, N, 384) == 0
    assert lb.lowbit_sa_packed_bytes(9, G, N, K) == 0
    # (P, G, M, K): G not in {64, 128, 256}; K not a multiple of 256; no planes; M > 32
    for P2, G2, M2, K2 in [(P, 32, 1, K), (P, G, 1, 384), (0, G, 1, K), (P, G, 33, K)]:
        with pytest.raises(lb.LowbitError) as e:
            lb.lowbit_gemm_sa(X, packed, P2, G2, M2, N, K2, Y)
        assert e.value.status == 2, (P2, G2, M2, K2)
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_sa_path(X, packed, P, G, 1, N, K, Y, 4)
    assert e.value.status == 1
