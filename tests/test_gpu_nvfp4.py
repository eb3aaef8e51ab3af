"""GPU parity for NVFP4 weights and the trimmed draft head (small-vocabulary MTP study, section
3.3: the head trimmed to 32,768 rows, quantised to NVFP4, winners mapped back to the full
vocabulary) through the C ABI against the CPU oracle (``oracle.nvfp4``)."""
import numpy as np
import pytest

import synth
from oracle import nvfp4 as onf
from oracle import verify as over
from helpers import bf16_dev, check_argmax, check_gemm, dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def pack_gpu(lb, codes, scales, g):
    N, KB = codes.shape
    K = KB * 2
    packed = torch.empty(lb.lowbit_nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_nvfp4(dev(codes), dev(scales), g, N, K, packed)
    return packed


def draft_gpu(lb, h, packed, M, N, K, ids_map, ws=None):
    if ws is None:
        ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    lb.lowbit_draft_argmax(bf16_dev(h), packed, M, N, K,
                           None if ids_map is None else dev(ids_map), out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ws


@pytest.mark.parametrize("N,K", [(1, 128), (257, 384), (128, 4096), (1000, 1024)])
def test_pack_nvfp4_bit_exact(lb, N, K):
    codes, scales, g, _, _ = synth.nvfp4_problem(40, 1, N, K)
    got = pack_gpu(lb, codes, scales, g).cpu().numpy()
    ref = onf.pack(codes, scales, g)
    assert got.shape == ref.shape and np.array_equal(got, ref)
    c2, s2, g2 = onf.unpack(got)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales) and g2 == np.float32(g)


@pytest.mark.parametrize("M", [1, 2, 16, 32])
@pytest.mark.parametrize("N,K", [(1, 128), (65, 256), (300, 1280), (2000, 512)])
def test_nvfp4_gemm_small_and_ragged(lb, N, K, M):
    codes, scales, g, _, x = synth.nvfp4_problem(41, M, N, K)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4(bf16_dev(x), pack_gpu(lb, codes, scales, g), M, N, K, Y)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y), onf.gemm(x, codes, scales, g), f"nvfp4 M={M} N={N} K={K}")


def test_nvfp4_subnormal_and_nan_scales(lb):
    """E4M3 subnormal scales decode exactly; a NaN scale makes its rows' outputs NaN."""
    M, N, K = 2, 256, 256
    codes, scales, g, _, x = synth.nvfp4_problem(42, M, N, K)
    scales = scales.copy()
    scales[:64] = synth.generator(43).integers(1, 8, size=(64, K // 16))  # exponent 0: subnormal
    scales[200, 3] = 0x7F
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4(bf16_dev(x), pack_gpu(lb, codes, scales, g), M, N, K, Y)
    torch.cuda.synchronize()
    y = host_bits(Y)
    from oracle import numerics
    assert np.isnan(numerics.bf16_to_f64(y[:, 200])).all()
    keep = np.array([n for n in range(N) if n != 200])
    check_gemm(y[:, keep], onf.gemm(x, codes[keep], scales[keep], g), "nvfp4 subnormal scales")


@pytest.mark.parametrize("with_map", [True, False])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 512), (4, 257, 256), (16, 3000, 1024), (32, 129, 128)])
def test_draft_argmax_small_and_planted(lb, M, N, K, with_map):
    codes, scales, g, ids, h = synth.nvfp4_problem(44, M, N, K)
    # plant a dominant row for token 0: codes +6 / -6 by the sign of each activation
    hv = (h.view(np.uint16)[0].astype(np.uint32) << 16).view(np.float32)
    c4 = np.where(hv > 0, 7, 15).astype(np.uint8)
    codes[N // 2] = c4[0::2] | (c4[1::2] << 4)
    scales[N // 2] = 0x48                                         # 2^(9-7) = 4
    logits = onf.gemm(h, codes, scales, g)
    assert over.argmax_lowest(logits)[0] == N // 2
    got, ws = draft_gpu(lb, h, pack_gpu(lb, codes, scales, g), M, N, K, ids if with_map else None)
    rows = np.searchsorted(ids, got) if with_map else got
    if with_map:
        assert np.array_equal(ids[rows], got)                      # every id is a mapped row
    assert rows[0] == N // 2
    check_argmax(rows, logits, f"draft M={M} N={N}")
    assert int(ws.sum().item()) == 0                               # workspace left zeroed


@pytest.mark.parametrize("M", [1, 16])
def test_draft_head_trimmed_full_size(lb, M):
    """The trimmed 32,768-row head at K = 4096: every argmax graded against the oracle, and the
    multiply itself on sampled rows."""
    N, K = synth.DRAFT_ROWS, synth.HEAD_K
    codes, scales, g, ids, h = synth.nvfp4_problem(4, M, N, K)
    packed = pack_gpu(lb, codes, scales, g)
    logits = onf.gemm(h, codes, scales, g)
    got, ws = draft_gpu(lb, h, packed, M, N, K, ids)
    check_argmax(np.searchsorted(ids, got), logits, f"trimmed head M={M}")
    assert np.array_equal(np.isin(got, ids), np.ones(M, dtype=bool))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4(bf16_dev(h), packed, M, N, K, Y)
    torch.cuda.synchronize()
    rows = np.sort(synth.generator(45, M).choice(N, size=2048, replace=False))
    check_gemm(host_bits(Y)[:, rows], logits[:, rows], f"trimmed head logits M={M}")


def test_draft_argmax_header_mismatch(lb):
    """An INT4 buffer passed as an NVFP4 head is rejected on the device; ids stay untouched."""
    N, K = 256, 512
    qc, qs, _ = synth.int4_problem(46, 1, N, K)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    from helpers import f16_dev
    lb.lowbit_pack_int4(dev(qc), f16_dev(qs), N, K, packed)
    lb.lowbit_device_error()
    _, _, _, _, h = synth.nvfp4_problem(46, 4, N, K)
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    out = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    lb.lowbit_draft_argmax(bf16_dev(h), packed, 4, N, K, None, out, ws)
    assert lb.lowbit_device_error() == 1
    assert bool((out == -7).all())


def test_draft_argmax_validation(lb):
    N, K = 64, 256
    codes, scales, g, ids, h = synth.nvfp4_problem(47, 1, N, K)
    packed = pack_gpu(lb, codes, scales, g)
    H = torch.zeros((33, K), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(33, dtype=torch.int32, device="cuda")
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_draft_argmax(H, packed, 33, N, K, None, out, ws)
    assert e.value.status == 2
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_draft_argmax(H, packed, 1, N, K, None, out, ws[:16])
    assert e.value.status == 4
    assert lb.lowbit_nvfp4_packed_bytes(N, 200) == 0
