"""GPU parity for Q8 weights and the 8-bit trimmed draft head (small-vocabulary MTP study,
section 3.3: the Q8 arm of its head comparison; w = d * q, int8 q, one fp16 d per 32 inputs)
through the C ABI against the CPU oracle (``oracle.q8``)."""
import numpy as np
import pytest

import synth
from oracle import q8 as oq8
from oracle import nvfp4 as onf
from oracle import verify as over
from helpers import Guarded, bf16_dev, check_argmax, check_gemm, dev, f16_dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def pack_gpu(lb, codes, scales):
    N, K = codes.shape
    packed = torch.empty(lb.lowbit_q8_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_q8(dev(codes), f16_dev(scales), N, K, packed)
    return packed


@pytest.mark.parametrize("N,K", [(1, 128), (257, 384), (128, 4096), (1000, 1024)])
def test_pack_q8_bit_exact(lb, N, K):
    codes, scales, _, _ = synth.q8_problem(70, 1, N, K)
    codes[0, :2] = (-128, 127)                                   # the full int8 range
    got = pack_gpu(lb, codes, scales).cpu().numpy()
    ref = oq8.pack(codes, scales)
    assert got.shape == ref.shape and np.array_equal(got, ref)
    c2, s2 = oq8.unpack(got)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)


@pytest.mark.parametrize("M", [1, 2, 4, 16, 32])
@pytest.mark.parametrize("N,K", [(1, 128), (65, 256), (300, 1280), (2000, 512), (129, 8192)])
def test_q8_gemm_small_ragged_and_deep(lb, N, K, M):
    codes, scales, _, x = synth.q8_problem(71, M, N, K)
    codes[:, :3] = (-128, 127, -127)                             # extreme codes on every row
    Y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    lb.lowbit_gemm_q8(bf16_dev(x), pack_gpu(lb, codes, scales), M, N, K, Y.t)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y.t), oq8.gemm(x, codes, scales), f"q8 M={M} N={N} K={K}")
    Y.check(f"q8 M={M}")


@pytest.mark.parametrize("N,K", [(300, 1024), (4096, 2048)])
def test_q8_m1_both_kernels(lb, N, K):
    """M = 1 on the streaming kernel (path 1) and on the warp-level MMA (path 3)."""
    codes, scales, _, x = synth.q8_problem(72, 1, N, K)
    ref = oq8.gemm(x, codes, scales)
    for path in (1, 3):
        Y = torch.full((1, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        lb.lowbit_gemm_q8_path(bf16_dev(x), pack_gpu(lb, codes, scales), 1, N, K, Y, path)
        torch.cuda.synchronize()
        check_gemm(host_bits(Y), ref, f"q8 M=1 path={path}")
    X2 = bf16_dev(np.repeat(x, 2, axis=0))
    Y2 = torch.empty((2, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LowbitError) as e:  # the streaming kernel takes one row
        lb.lowbit_gemm_q8_path(X2, pack_gpu(lb, codes, scales), 2, N, K, Y2, 1)
    assert e.value.status == 2


@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("kind", synth.ACTIVATION_KINDS)
def test_q8_activation_structures(lb, kind, M):
    """Outliers, mixed magnitudes per 64 inputs, 2^-90 / 2^90 magnitudes (compared after an
    exact power-of-two rescaling), zeros and sparse activations."""
    N, K = 260, 1024
    g = synth.generator(73, synth.ACTIVATION_KINDS.index(kind), M)
    codes, scales = synth.q8_weights(g, N, K)
    x = synth.activation_variant(g, M, K, kind)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_q8(bf16_dev(x), pack_gpu(lb, codes, scales), M, N, K, Y)
    torch.cuda.synchronize()
    scale = {"tiny": 2.0 ** 90, "huge": 2.0 ** -90}.get(kind, 1.0)
    check_gemm(host_bits(Y), oq8.gemm(x, codes, scales), f"q8 {kind} M={M}", scale=scale)


@pytest.mark.parametrize("with_map", [True, False])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 512), (1, 129, 8192), (4, 257, 256), (16, 3000, 1024),
                                   (32, 129, 128)])
def test_q8_draft_argmax_small_and_planted(lb, M, N, K, with_map):
    codes, scales, ids, h = synth.q8_problem(74, M, N, K)
    hv = (h.view(np.uint16)[0].astype(np.uint32) << 16).view(np.float32)
    codes[N // 2] = np.where(hv > 0, 127, -127).astype(np.int8)   # a dominant row for token 0
    scales[N // 2] = synth.to_f16_bits(np.full(K // 32, 0.01))
    logits = oq8.gemm(h, codes, scales)
    assert over.argmax_lowest(logits)[0] == N // 2
    ws = Guarded((lb.lmhead_workspace_bytes(2, N, K),), torch.uint8, fill=0)
    out = Guarded((M,), torch.int32, fill=-1)
    lb.lowbit_draft_argmax_q8(bf16_dev(h), pack_gpu(lb, codes, scales), M, N, K,
                              dev(ids) if with_map else None, out.t, ws.t)
    torch.cuda.synchronize()
    got = out.t.cpu().numpy()
    rows = np.searchsorted(ids, got) if with_map else got
    if with_map:
        assert np.array_equal(ids[rows], got)                      # every id is a mapped row
    assert rows[0] == N // 2
    check_argmax(rows, logits, f"q8 draft M={M} N={N}")
    assert not ws.t.any()                                          # workspace left zeroed
    ws.check("q8 draft workspace")
    out.check("q8 draft ids")


@pytest.mark.parametrize("M", [1, 16])
def test_q8_trimmed_head_full_size(lb, M):
    """The trimmed 32,768-row head at K = 4096: every argmax graded against the oracle, and the
    logits of sampled rows."""
    N, K = synth.DRAFT_ROWS, synth.HEAD_K
    codes, scales, ids, h = synth.q8_problem(4, M, N, K)
    packed = pack_gpu(lb, codes, scales)
    logits = oq8.gemm(h, codes, scales)
    ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    lb.lowbit_draft_argmax_q8(bf16_dev(h), packed, M, N, K, dev(ids), out, ws)
    torch.cuda.synchronize()
    check_argmax(np.searchsorted(ids, out.cpu().numpy()), logits, f"q8 trimmed head M={M}")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_q8(bf16_dev(h), packed, M, N, K, Y)
    torch.cuda.synchronize()
    rows = np.arange(0, N, 97)
    check_gemm(host_bits(Y)[:, rows], logits[:, rows], f"q8 trimmed head logits M={M}")
    assert lb.lowbit_device_error() == 0


def test_q8_header_mismatch_is_recorded_and_writes_nothing(lb):
    N, K = 300, 512
    codes, scales, _, x = synth.q8_problem(75, 1, N, K)
    packed = pack_gpu(lb, codes, scales)
    lb.lowbit_device_error()
    for M in (1, 16):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        lb.lowbit_gemm_q8(bf16_dev(np.repeat(x, M, axis=0)), packed, M, N, 256, Y)  # wrong K
        torch.cuda.synchronize()
        assert lb.lowbit_device_error() == 1
        assert torch.isnan(Y.float()).all()
