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


def draft_gpu(lb, h, packed, M, N, K, ids_map, ws=None, path=0):
    if ws is None:
        ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    out = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    lb.lowbit_draft_argmax_path(bf16_dev(h), packed, M, N, K,
                                None if ids_map is None else dev(ids_map), out, ws, path)
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


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("N,K", [(1, 128), (127, 256), (129, 4096), (300, 8192), (1000, 1152),
                                 (4096, 2048)])
def test_nvfp4_m1_both_paths(lb, N, K, path):
    """M = 1 on the streaming mat-vec (path 1) and on the tensor cores (path 2); the shapes span
    one row tile, ragged tiles, deep K splits (few tiles, long K) and many tiles."""
    codes, scales, g, _, x = synth.nvfp4_problem(48, 1, N, K)
    Y = torch.full((1, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4_path(bf16_dev(x), pack_gpu(lb, codes, scales, g), 1, N, K, Y, path)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y), onf.gemm(x, codes, scales, g), f"nvfp4 M=1 N={N} K={K} path={path}")


@pytest.mark.parametrize("kind", ("outlier", "mixed_scale", "tiny", "sparse"))
def test_nvfp4_m1_activation_structures(lb, kind):
    """The streaming path's int16 activations (one power-of-two scale per 64 inputs) under
    outliers, mixed magnitudes, tiny values and zero runs."""
    N, K = 260, 1024
    g = synth.generator(49, synth.ACTIVATION_KINDS.index(kind))
    codes, scales, gs = synth.nvfp4_weights(g, N, K)
    x = synth.activation_variant(g, 1, K, kind)
    Y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4_path(bf16_dev(x), pack_gpu(lb, codes, scales, gs), 1, N, K, Y, 1)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y), onf.gemm(x, codes, scales, gs), f"nvfp4 {kind}",
               scale=2.0 ** 90 if kind == "tiny" else 1.0)


@pytest.mark.parametrize("M,path", [(1, 1), (2, 2)])
def test_nvfp4_subnormal_and_nan_scales(lb, M, path):
    """E4M3 subnormal scales decode exactly; a NaN scale makes its rows' outputs NaN."""
    N, K = 256, 256
    codes, scales, g, _, x = synth.nvfp4_problem(42, M, N, K)
    scales = scales.copy()
    scales[:64] = synth.generator(43).integers(1, 8, size=(64, K // 16))  # exponent 0: subnormal
    scales[200, 3] = 0x7F
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4_path(bf16_dev(x), pack_gpu(lb, codes, scales, g), M, N, K, Y, path)
    torch.cuda.synchronize()
    y = host_bits(Y)
    from oracle import numerics
    assert np.isnan(numerics.bf16_to_f64(y[:, 200])).all()
    keep = np.array([n for n in range(N) if n != 200])
    check_gemm(y[:, keep], onf.gemm(x, codes[keep], scales[keep], g), "nvfp4 subnormal scales")


@pytest.mark.parametrize("with_map", [True, False])
@pytest.mark.parametrize("M,N,K,path", [(1, 1000, 512, 1), (1, 1000, 512, 2), (1, 129, 8192, 1),
                                        (4, 257, 256, 0), (16, 3000, 1024, 0), (32, 129, 128, 0)])
def test_draft_argmax_small_and_planted(lb, M, N, K, path, with_map):
    codes, scales, g, ids, h = synth.nvfp4_problem(44, M, N, K)
    # plant a dominant row for token 0: codes +6 / -6 by the sign of each activation
    hv = (h.view(np.uint16)[0].astype(np.uint32) << 16).view(np.float32)
    c4 = np.where(hv > 0, 7, 15).astype(np.uint8)
    codes[N // 2] = c4[0::2] | (c4[1::2] << 4)
    scales[N // 2] = 0x48                                         # 2^(9-7) = 4
    logits = onf.gemm(h, codes, scales, g)
    assert over.argmax_lowest(logits)[0] == N // 2
    got, ws = draft_gpu(lb, h, pack_gpu(lb, codes, scales, g), M, N, K, ids if with_map else None,
                        path=path)
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


@pytest.mark.parametrize("M", [1, 4])
def test_draft_argmax_header_mismatch(lb, M):
    """An INT4 buffer passed as an NVFP4 head is rejected on the device; ids stay untouched and
    the workspace stays zero (no CTA counts itself in)."""
    N, K = 1000, 512
    qc, qs, _ = synth.int4_problem(46, 1, N, K)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    from helpers import f16_dev
    lb.lowbit_pack_int4(dev(qc), f16_dev(qs), N, K, packed)
    lb.lowbit_device_error()
    _, _, _, _, h = synth.nvfp4_problem(46, M, N, K)
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    out = torch.full((M,), -7, dtype=torch.int32, device="cuda")
    lb.lowbit_draft_argmax(bf16_dev(h), packed, M, N, K, None, out, ws)
    assert lb.lowbit_device_error() == 1
    assert bool((out == -7).all())
    assert int(ws.sum().item()) == 0
    Y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_nvfp4(bf16_dev(h), packed, M, N, K, Y)
    assert lb.lowbit_device_error() == 1
    assert bool((Y == 7.0).all())


def test_draft_argmax_m1_back_to_back(lb):
    """Recursive drafting: successive M = 1 calls on one stream share one workspace; each call
    sees only its own keys (the next launch may start before the previous one has reset the
    workspace, and must wait for it)."""
    N, K = 4096, 1024
    codes, scales, g, ids, _ = synth.nvfp4_problem(50, 1, N, K)
    packed = pack_gpu(lb, codes, scales, g)
    hs = [synth.nvfp4_problem(51 + i, 1, N, K)[4] for i in range(8)]
    ws = torch.zeros(lb.lmhead_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    outs = [torch.full((1,), -1, dtype=torch.int32, device="cuda") for _ in hs]
    hd = [bf16_dev(h) for h in hs]
    imap = dev(ids)
    for h, o in zip(hd, outs):
        lb.lowbit_draft_argmax(h, packed, 1, N, K, imap, o, ws)
    torch.cuda.synchronize()
    for h, o in zip(hs, outs):
        row = np.searchsorted(ids, o.cpu().numpy())
        check_argmax(row, onf.gemm(h, codes, scales, g), "back-to-back draft")
    assert int(ws.sum().item()) == 0


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
    with pytest.raises(lb.LowbitError) as e:                       # streaming path: M = 1 only
        lb.lowbit_draft_argmax_path(H, packed, 2, N, K, None, out, ws, 1)
    assert e.value.status == 2
    Y = torch.empty((2, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_nvfp4_path(H, packed, 2, N, K, Y, 1)
    assert e.value.status == 2
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_nvfp4_path(H, packed, 1, N, K, Y, 3)
    assert e.value.status == 1
    assert lb.lowbit_nvfp4_packed_bytes(N, 200) == 0
