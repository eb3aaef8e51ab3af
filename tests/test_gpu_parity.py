"""GPU parity: every hot-path row through the C ABI against the CPU oracle.

Inputs come from the seeded generators in ``synth``; expected values come only from
``oracle``.  Sizes span several row tiles and a ragged tail; the full workload shapes are
checked too (all outputs where the oracle finishes in seconds)."""
import numpy as np
import pytest

import synth
from oracle import binplane as obp
from oracle import int4 as oint4
from oracle import verify as over
from helpers import bf16_dev, check_argmax, check_gemm, dev, f16_dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def pack_int4_gpu(lb, codes, scales):
    N, K = codes.shape
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, packed)
    return packed


def pack_bp_gpu(lb, bits, alpha):
    P, N, KB = bits.shape
    K = KB * 8
    packed = torch.empty(lb.lowbit_binplane_packed_bytes(P, N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_binplane(dev(bits), f16_dev(alpha), P, N, K, packed)
    return packed


def gemm_int4_gpu(lb, x, packed, M, N, K, path=0):
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_int4_path(bf16_dev(x), packed, M, N, K, Y, path)
    torch.cuda.synchronize()
    return host_bits(Y)


def gemm_bp_gpu(lb, x, packed, P, M, N, K, path=0):
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_binplane_path(bf16_dev(x), packed, P, M, N, K, Y, path)
    torch.cuda.synchronize()
    return host_bits(Y)


PATHS = (1, 2)   # 1 = CUDA-core kernels, 2 = tensor-core kernels (tcgen05)
INT4_PATHS = (1, 2, 3)   # INT4, binary planes and the LM head also: 3 = warp-level MMA kernels


# ------------------------------------------------------------------------- packing

@pytest.mark.parametrize("N,K", [(256, 512), (257, 384), (8, 128), (1, 128), (4096, 2560),
                                 (2560, 9728)])
def test_pack_int4_bit_exact(lb, N, K):
    codes, scales, _ = synth.int4_problem(0, 1, N, K, 77)
    got = pack_int4_gpu(lb, codes, scales).cpu().numpy()
    ref = oint4.pack(codes, scales)
    assert got.shape == ref.shape and np.array_equal(got, ref)
    c2, s2 = oint4.unpack(got)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    assert lb.lowbit_validate_packed(pack_int4_gpu(lb, codes, scales), 1, 0, N, K) == 0
    assert lb.lowbit_validate_packed(pack_int4_gpu(lb, codes, scales), 1, 0, N + 1, K) == 1


@pytest.mark.parametrize("P,N,K", [(3, 64, 256), (4, 33, 128), (1, 300, 512), (3, 12288, 4096),
                                   (4, 4096, 12288)])
def test_pack_binplane_bit_exact(lb, P, N, K):
    bits, alpha, _ = synth.binplane_problem(3, P, 1, N, K, 78)
    got = pack_bp_gpu(lb, bits, alpha).cpu().numpy()
    ref = obp.pack(bits, alpha)
    assert np.array_equal(got, ref)
    b2, a2 = obp.unpack(got)
    assert np.array_equal(b2, bits) and np.array_equal(a2, alpha)


# ------------------------------------------------------------------------- INT4 GEMV / GEMM

@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (1, 257, 384), (1, 1, 128), (1, 8, 1024),
                                   (1, 100, 12288), (2, 96, 256), (3, 65, 640), (16, 300, 1280),
                                   (32, 33, 384), (5, 1, 128), (17, 129, 2048), (16, 2000, 256)])
def test_int4_small_and_ragged(lb, M, N, K, path):
    codes, scales, x = synth.int4_problem(0, M, N, K)
    packed = pack_int4_gpu(lb, codes, scales)
    y = gemm_int4_gpu(lb, x, packed, M, N, K, path)
    check_gemm(y, oint4.gemm(x, codes, scales), f"int4 M={M} N={N} K={K} path={path}")


ACT_SCALE = {"tiny": 2.0 ** 90, "huge": 2.0 ** -90}


@pytest.mark.parametrize("M,path", [(1, 1), (16, 1), (16, 2), (16, 3), (32, 3)])
@pytest.mark.parametrize("kind", synth.ACTIVATION_KINDS)
def test_int4_activation_structures(lb, kind, M, path):
    """Outlier channels, per-run magnitude swings, extreme exponents, zeros and sparsity: the
    M = 1 kernel holds each run of 64 activations as int16 under one power of two, so these
    are the inputs that would expose a lost scale, a clipped outlier or a rounding bias."""
    N, K = 645, 1408
    g = synth.generator(91, M, N, K, synth.ACTIVATION_KINDS.index(kind))
    codes, scales = synth.int4_weights(g, N, K)
    x = synth.activation_variant(g, M, K, kind)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), M, N, K, path)
    check_gemm(y, oint4.gemm(x, codes, scales), f"int4 {kind} M={M} path={path}",
               scale=ACT_SCALE.get(kind, 1.0))


@pytest.mark.parametrize("M,path", [(1, 1), (16, 1), (16, 2), (16, 3), (32, 3)])
def test_int4_nan_activation(lb, M, path):
    """A NaN activation in token 0 makes token 0's outputs NaN and leaves the others exact."""
    N, K = 300, 640
    codes, scales, x = synth.int4_problem(92, M, N, K)
    x = x.copy()
    x[0, 333] = 0x7FC0
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), M, N, K, path)
    from oracle import numerics
    assert np.isnan(numerics.bf16_to_f64(y[0])).all()
    if M > 1:
        check_gemm(y[1:], oint4.gemm(x[1:], codes, scales), f"int4 NaN rows 1.. path={path}")


@pytest.mark.parametrize("M,path", [(1, 1), (16, 2), (16, 3)])
@pytest.mark.parametrize("kind", ("outlier", "mixed_scale", "tiny", "sparse"))
def test_binplane_activation_structures(lb, kind, M, path):
    P, N, K = 3, 260, 1024
    g = synth.generator(93, P, M, N, K, synth.ACTIVATION_KINDS.index(kind))
    bits, alpha = synth.binplane_weights(g, P, N, K)
    x = synth.activation_variant(g, M, K, kind)
    y = gemm_bp_gpu(lb, x, pack_bp_gpu(lb, bits, alpha), P, M, N, K, path)
    check_gemm(y, obp.gemm(x, bits, alpha), f"binplane {kind} M={M} path={path}",
               scale=ACT_SCALE.get(kind, 1.0))


@pytest.mark.parametrize("N,K", [(5000, 5120), (4864, 8192)])
def test_int4_m1_ring_at_default_smem_limit(lb, N, K):
    """Shapes whose ring plus split-K slots (about 46-48 KB) fit under 48 KB while ring plus
    the kernel's static shared memory does not: the launch needs the large-shared-memory
    opt-in even though the dynamic size alone is below 48 KB."""
    codes, scales, x = synth.int4_problem(94, 1, N, K)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), 1, N, K)
    check_gemm(y, oint4.gemm(x, codes, scales), f"int4 M=1 N={N} K={K}")


@pytest.mark.parametrize("P,N,K", [(5, 200, 5120), (5, 1300, 5120)])
def test_binplane_m1_ring_at_default_smem_limit(lb, P, N, K):
    bits, alpha, x = synth.binplane_problem(95, P, 1, N, K)
    y = gemm_bp_gpu(lb, x, pack_bp_gpu(lb, bits, alpha), P, 1, N, K, 1)
    check_gemm(y, obp.gemm(x, bits, alpha), f"binplane M=1 P={P} N={N} K={K}")


def test_int4_tiny_gemv(lb):
    cfg = synth.WORKLOADS["tiny"]
    (K, N), = cfg["shapes"]
    codes, scales, x = synth.int4_problem(cfg["seed"], 1, N, K)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), 1, N, K)
    check_gemm(y, oint4.gemm(x, codes, scales), "tiny GEMV")


@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("proj", range(7))
def test_int4_decode_layer(lb, proj, path):
    cfg = synth.WORKLOADS["decode"]
    K, N = cfg["shapes"][proj]
    codes, scales, x = synth.int4_problem(cfg["seed"], 1, N, K, proj)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), 1, N, K, path)
    check_gemm(y, oint4.gemm(x, codes, scales), f"decode layer proj {proj} path={path}")


@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("M", synth.M_SWEEP)
@pytest.mark.parametrize("proj", [0, 1, 6])
def test_int4_verify_layer_m_sweep(lb, proj, M, path):
    cfg = synth.WORKLOADS["verify"]
    K, N = cfg["shapes"][proj]
    codes, scales, x = synth.int4_problem(cfg["seed"], M, N, K, proj)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), M, N, K, path)
    check_gemm(y, oint4.gemm(x, codes, scales), f"verify layer proj {proj} M={M} path={path}")


@pytest.mark.parametrize("proj", [2, 3, 4, 5])
def test_int4_verify_layer_remaining_projections(lb, proj):
    cfg = synth.WORKLOADS["verify"]
    K, N = cfg["shapes"][proj]
    codes, scales, x = synth.int4_problem(cfg["seed"], 16, N, K, proj)
    y = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), 16, N, K)
    check_gemm(y, oint4.gemm(x, codes, scales), f"verify layer proj {proj}")


# ------------------------------------------------------------------------- binary planes

@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("P,M,N,K", [(3, 1, 64, 256), (4, 2, 33, 128), (1, 16, 300, 512),
                                     (2, 5, 8, 1024), (3, 32, 40, 384), (8, 20, 130, 640)])
def test_binplane_small_and_ragged(lb, P, M, N, K, path):
    bits, alpha, x = synth.binplane_problem(3, P, M, N, K)
    packed = pack_bp_gpu(lb, bits, alpha)
    y = gemm_bp_gpu(lb, x, packed, P, M, N, K, path)
    check_gemm(y, obp.gemm(x, bits, alpha), f"binplane P={P} M={M} N={N} K={K} path={path}")


@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("shape", [0, 1])
@pytest.mark.parametrize("P", synth.BINPLANE_PLANES)
@pytest.mark.parametrize("M", (1, 16))
def test_binplane_matrices(lb, shape, P, M, path):
    cfg = synth.WORKLOADS["binplane"]
    K, N = cfg["shapes"][shape]
    bits, alpha, x = synth.binplane_problem(cfg["seed"], P, M, N, K, shape)
    packed = pack_bp_gpu(lb, bits, alpha)
    y = gemm_bp_gpu(lb, x, packed, P, M, N, K, path)
    check_gemm(y, obp.gemm(x, bits, alpha), f"binary planes K={K} N={N} P={P} M={M} path={path}")


# ------------------------------------------------------------------------- LM head verify

def run_lmhead(lb, h, packed, M, N, K, drafts, ws=None, path=0):
    if ws is None:
        ws = torch.zeros(lb.lmhead_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    a = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    b = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lb.lmhead_argmax_verify_path(bf16_dev(h), packed, M, N, K, dev(drafts.astype(np.int32)), a, n,
                                 b, ws, path)
    torch.cuda.synchronize()
    return a.cpu().numpy(), int(n.item()), int(b.item()), ws


def check_lmhead(a, n, b, logits, drafts, j, what):
    check_argmax(a, logits, what)
    # acceptance is bit-exact against the prefix rule on the GPU's own argmax ...
    assert (n, b) == over.accept(a, drafts), what
    # ... and equals the planted j whenever rows 0..j are decided by a clear margin
    margin = over.top2_margin(logits)
    if np.all(margin[: j + 1] > 1e-2):
        assert n == j, what


@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("rows", synth.HEAD_ROWS)
def test_lmhead_full_and_trimmed_heads(lb, rows, path):
    cfg = synth.WORKLOADS["lmhead"]
    M, K = cfg["M"], cfg["K"]
    codes, scales, h = synth.int4_problem(cfg["seed"], M, rows, K)
    packed = pack_int4_gpu(lb, codes, scales)
    logits = oint4.gemm(h, codes, scales)
    a_ref = over.argmax_lowest(logits)
    ws = None
    for trial, j in enumerate((None, 0, 15)):
        drafts, jj = synth.plant_drafts(cfg["seed"] + trial, a_ref, rows, j)
        a, n, b, ws = run_lmhead(lb, h, packed, M, rows, K, drafts, ws, path)
        check_lmhead(a, n, b, logits, drafts, jj, f"LM head N={rows} j={jj}")
    # the workspace is left zeroed for the next call
    assert int(ws.sum().item()) == 0


@pytest.mark.parametrize("path", INT4_PATHS)
@pytest.mark.parametrize("M,N,K", [(2, 40, 128), (16, 1000, 512), (32, 257, 256), (7, 5, 128),
                                   (16, 300, 2048)])
def test_lmhead_small_and_planted(lb, M, N, K, path):
    codes, scales, h = synth.int4_problem(11, M, N, K)
    # plant a dominant row for token 0 so at least one row is decided by construction
    hv = h.view(np.uint16)
    xv = (hv[0].astype(np.uint32) << 16).view(np.float32)
    codes[N // 2] = np.where(xv > 0, 7, -8)
    scales[N // 2] = np.float16(1.0).view(np.uint16)
    logits = oint4.gemm(h, codes, scales)
    a_ref = over.argmax_lowest(logits)
    assert a_ref[0] == N // 2
    drafts, j = synth.plant_drafts(2, a_ref, N)
    a, n, b, _ = run_lmhead(lb, h, pack_int4_gpu(lb, codes, scales), M, N, K, drafts, path=path)
    assert a[0] == N // 2
    check_lmhead(a, n, b, logits, drafts, j, f"lmhead M={M} N={N}")


# ------------------------------------------------------------------------- error paths

@pytest.mark.parametrize("path", INT4_PATHS)
def test_header_mismatch_is_recorded_and_nothing_written(lb, path):
    codes, scales, x = synth.int4_problem(1, 1, 64, 256)
    packed = pack_int4_gpu(lb, codes, scales)
    assert lb.lowbit_device_error() == 0
    Y = torch.full((1, 96), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_int4_path(bf16_dev(x), packed, 1, 96, 256, Y, path)   # header says N = 64
    assert lb.lowbit_device_error() == 1
    assert torch.all(Y == 7.0)
    assert lb.lowbit_device_error() == 0                        # cleared by the read


@pytest.mark.parametrize("path", INT4_PATHS)
def test_header_mismatch_beyond_the_allocation(lb, path):
    """A claimed shape whose payload cannot lie inside the buffer's allocation: the kernels
    check the header before reading any weight, record the mismatch and write nothing."""
    codes, scales, x = synth.int4_problem(1, 1, 64, 256)
    packed = pack_int4_gpu(lb, codes, scales)                  # 17 KB
    N = 65536                                                  # claims 8.6 MB of payload
    Y = torch.full((1, N), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_int4_path(bf16_dev(x), packed, 1, N, 256, Y, path)
    assert lb.lowbit_device_error() == 1
    assert torch.all(Y == 7.0)


@pytest.mark.parametrize("N", [96, 65536])
def test_binplane_header_mismatch_is_recorded_and_nothing_written(lb, N):
    bits, alpha, x = synth.binplane_problem(3, 3, 1, 64, 256, 5)
    packed = pack_bp_gpu(lb, bits, alpha)
    assert lb.lowbit_device_error() == 0
    Y = torch.full((1, N), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_binplane(bf16_dev(x), packed, 3, 1, N, 256, Y)
    assert lb.lowbit_device_error() == 1
    assert torch.all(Y == 7.0)
    # a plane count that disagrees with the header is caught the same way
    Y2 = torch.full((1, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lb.lowbit_gemm_binplane(bf16_dev(x), packed, 2, 1, 64, 256, Y2)
    assert lb.lowbit_device_error() == 1
    assert torch.all(Y2 == 7.0)


def test_shape_errors_raise(lb):
    codes, scales, x = synth.int4_problem(1, 1, 64, 256)
    packed = pack_int4_gpu(lb, codes, scales)
    Y = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_int4(bf16_dev(x), packed, 1, 64, 200, Y)
    assert e.value.status == 2


# ------------------------------------------------------------------------- grouped multiplies

def _grouped(lb, M, shapes, seed, path=0):
    probs, refs = [], []
    for j, (K, N) in enumerate(shapes):
        codes, scales, x = synth.int4_problem(seed, M, N, K, j)
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        probs.append((bf16_dev(x), pack_int4_gpu(lb, codes, scales), N, K, Y))
        refs.append(oint4.gemm(x, codes, scales))
    if path:
        lb.lowbit_gemm_int4_grouped_path(probs, M, path)
    else:
        lb.lowbit_gemm_int4_grouped(probs, M)
    torch.cuda.synchronize()
    return [host_bits(p[4]) for p in probs], refs


@pytest.mark.parametrize("M", [1, 16])
def test_grouped_decode_layer_in_one_call(lb, M):
    """The seven projections of the 4B-class layer as one grouped call (one launch at M=1)."""
    shapes = synth.WORKLOADS["decode"]["shapes"]
    ys, refs = _grouped(lb, M, shapes, synth.WORKLOADS["decode"]["seed"] if M == 1 else synth.WORKLOADS["verify"]["seed"])
    for j, (y, r) in enumerate(zip(ys, refs)):
        check_gemm(y, r, f"grouped M={M} proj {j}")


@pytest.mark.parametrize("shapes", [
    ((512, 256),),
    ((384, 257), (128, 1), (1280, 300)),
    ((2560, 4096), (2560, 1024), (2560, 1024)),          # q, k, v share one launch
    ((2560, 9728), (2560, 9728)),                        # gate, up
    ((12288, 100), (128, 8), (256, 129), (640, 65), (128, 2), (1024, 33), (384, 1000), (896, 7)),
])
@pytest.mark.parametrize("M,path", [(1, 0), (2, 0), (16, 0), (32, 0), (16, 2), (32, 2), (4, 1),
                                    (3, 3)])
def test_grouped_ragged_mixes(lb, shapes, M, path):
    ys, refs = _grouped(lb, M, shapes, 11, path)
    for j, (y, r) in enumerate(zip(ys, refs)):
        check_gemm(y, r, f"grouped M={M} path={path} mix {shapes} item {j}")


def test_grouped_matches_single_calls_bit_for_bit(lb):
    """A matrix gives the same bf16 outputs alone and inside a group (same K split)."""
    shapes = ((2560, 1024), (2560, 1024))
    ys, _ = _grouped(lb, 1, shapes, 12)
    codes, scales, x = synth.int4_problem(12, 1, 1024, 2560, 0)
    y1 = gemm_int4_gpu(lb, x, pack_int4_gpu(lb, codes, scales), 1, 1024, 2560, 1)
    check_gemm(y1, oint4.gemm(x, codes, scales), "single")
    assert np.array_equal(ys[0], y1)


def test_grouped_validation(lb):
    codes, scales, x = synth.int4_problem(0, 1, 64, 256)
    X, P = bf16_dev(x), pack_int4_gpu(lb, codes, scales)
    Y = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_int4_grouped([(X, P, 64, 256, Y)] * 9, 1)
    assert e.value.status == 1
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_int4_grouped([(X, P, 64, 256, Y), (X, P, 64, 100, Y)], 1)
    assert e.value.status == 2
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_int4_grouped([], 1)
    assert e.value.status == 1

