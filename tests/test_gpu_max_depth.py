"""GPU parity at the deepest reduction the library accepts (K = 65,536 inputs) for every weight
format, every kernel family and the fused heads.

At this depth the schedulers hit their split-K ceiling (16 CTAs per row tile), so each CTA
streams the most blocks it ever does; the M = 1 kernels convert 1,024 runs of 64 activations
and the tensor-core kernels chain the longest accumulation in TMEM.  N = 1 (one tile, all
depth) and N = 257 (three tiles, a ragged tail) bracket the row layouts.  Outputs are written
into canary-banded buffers, so a write past either end is caught too."""
import numpy as np
import pytest

import synth
from oracle import binplane as obp
from oracle import int4 as oint4
from oracle import nvfp4 as onf
from oracle import q8 as oq8
from oracle import sa as osa
from oracle import verify as over
from helpers import Guarded, bf16_dev, check_argmax, check_gemm, dev, f16_dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

K_MAX = 65536


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def out_buf(M, N):
    return Guarded((M, N), torch.bfloat16, fill=float("nan"))


def finish(Y, Y64, what):
    torch.cuda.synchronize()
    check_gemm(host_bits(Y.t), Y64, what)
    Y.check(what)


def test_k_limit_is_enforced(lb):
    """One group past the limit is a shape error, raised before anything is enqueued."""
    N, K = 8, K_MAX + 64
    X = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    Y = torch.full((1, N), 7.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LowbitError) as e:
        lb.lowbit_gemm_int4(X, packed, 1, N, K, Y)
    assert e.value.status == 2
    assert torch.all(Y == 7.0)


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("N", [1, 257])
def test_int4_k_max(lb, N, M, path):
    codes, scales, x = synth.int4_problem(120, M, N, K_MAX)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K_MAX, packed)
    Y = out_buf(M, N)
    lb.lowbit_gemm_int4_path(bf16_dev(x), packed, M, N, K_MAX, Y.t, path)
    finish(Y, oint4.gemm(x, codes, scales), f"int4 K=65536 N={N} M={M} path={path}")


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("P,N", [(3, 257), (1, 1)])
def test_binplane_k_max(lb, P, N, M, path):
    bits, alpha, x = synth.binplane_problem(121, P, M, N, K_MAX)
    packed = torch.empty(lb.lowbit_binplane_packed_bytes(P, N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_binplane(dev(bits), f16_dev(alpha), P, N, K_MAX, packed)
    Y = out_buf(M, N)
    lb.lowbit_gemm_binplane_path(bf16_dev(x), packed, P, M, N, K_MAX, Y.t, path)
    finish(Y, obp.gemm(x, bits, alpha), f"binplane K=65536 P={P} N={N} M={M} path={path}")


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("P,G,N", [(2, 128, 257), (3, 64, 1)])
def test_sa_k_max(lb, P, G, N, M, path):
    bits, codes, d, x = synth.sa_problem(122, P, G, M, N, K_MAX)
    packed = torch.empty(lb.lowbit_sa_packed_bytes(P, G, N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_sa(dev(bits), dev(codes), f16_dev(d), P, G, N, K_MAX, packed)
    Y = out_buf(M, N)
    lb.lowbit_gemm_sa_path(bf16_dev(x), packed, P, G, M, N, K_MAX, Y.t, path)
    finish(Y, osa.gemm(x, bits, codes, d, G), f"sa K=65536 P={P} G={G} N={N} M={M} path={path}")


def pack_nvfp4(lb, codes, scales, g, N):
    packed = torch.empty(lb.lowbit_nvfp4_packed_bytes(N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_nvfp4(dev(codes), dev(scales), g, N, K_MAX, packed)
    return packed


@pytest.mark.parametrize("M,path", [(1, 1), (1, 2), (16, 0), (32, 0)])
@pytest.mark.parametrize("N", [1, 257])
def test_nvfp4_k_max(lb, N, M, path):
    codes, scales, g, _, x = synth.nvfp4_problem(123, M, N, K_MAX)
    Y = out_buf(M, N)
    lb.lowbit_gemm_nvfp4_path(bf16_dev(x), pack_nvfp4(lb, codes, scales, g, N), M, N, K_MAX, Y.t, path)
    finish(Y, onf.gemm(x, codes, scales, g), f"nvfp4 K=65536 N={N} M={M} path={path}")


def pack_q8(lb, codes, scales, N):
    packed = torch.empty(lb.lowbit_q8_packed_bytes(N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_q8(dev(codes), f16_dev(scales), N, K_MAX, packed)
    return packed


@pytest.mark.parametrize("M,path", [(1, 1), (1, 3), (16, 0), (32, 0)])
@pytest.mark.parametrize("N", [1, 257])
def test_q8_k_max(lb, N, M, path):
    codes, scales, _, x = synth.q8_problem(124, M, N, K_MAX)
    codes[:, :2] = (-128, 127)
    Y = out_buf(M, N)
    lb.lowbit_gemm_q8_path(bf16_dev(x), pack_q8(lb, codes, scales, N), M, N, K_MAX, Y.t, path)
    finish(Y, oq8.gemm(x, codes, scales), f"q8 K=65536 N={N} M={M} path={path}")


def plant_row(codes_like, h, row, hi, lo):
    """Make ``row`` dominant for token 0: each weight takes the sign of that token's input."""
    xv = (h.view(np.uint16)[0].astype(np.uint32) << 16).view(np.float32)
    codes_like[row] = np.where(xv > 0, hi, lo)


@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("M", [2, 16])
def test_lmhead_verify_k_max(lb, M, path):
    """Argmax over 1,000 rows at K = 65,536 and the greedy acceptance on the GPU's argmax."""
    N = 1000
    codes, scales, h = synth.int4_problem(125, M, N, K_MAX)
    plant_row(codes, h, 617, 7, -8)
    scales[617] = np.float16(1.0).view(np.uint16)
    logits = oint4.gemm(h, codes, scales)
    a_ref = over.argmax_lowest(logits)
    assert a_ref[0] == 617
    drafts, j = synth.plant_drafts(126, a_ref, N)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K_MAX), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K_MAX, packed)
    ws = torch.zeros(lb.lmhead_workspace_bytes(M, N, K_MAX), dtype=torch.uint8, device="cuda")
    a = Guarded((M,), torch.int32, fill=-1)
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    b = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lb.lmhead_argmax_verify_path(bf16_dev(h), packed, M, N, K_MAX, dev(drafts.astype(np.int32)),
                                 a.t, n, b, ws, path)
    torch.cuda.synchronize()
    got = a.t.cpu().numpy()
    assert got[0] == 617
    check_argmax(got, logits, f"lmhead K=65536 M={M} path={path}")
    assert (int(n.item()), int(b.item())) == over.accept(got, drafts)
    assert int(ws.sum().item()) == 0
    a.check("lmhead argmax")


@pytest.mark.parametrize("fmt", ["nvfp4", "q8"])
@pytest.mark.parametrize("M", [1, 16])
def test_draft_head_k_max(lb, fmt, M):
    """The trimmed draft heads at K = 65,536, winners mapped to full-vocabulary ids."""
    N = 1000
    if fmt == "nvfp4":
        codes, scales, g, ids, h = synth.nvfp4_problem(127, M, N, K_MAX)
        logits = onf.gemm(h, codes, scales, g)
        packed = pack_nvfp4(lb, codes, scales, g, N)
        call = lb.lowbit_draft_argmax
    else:
        codes, scales, ids, h = synth.q8_problem(127, M, N, K_MAX)
        plant_row(codes, h, 389, 127, -127)
        scales[389] = synth.to_f16_bits(np.full(K_MAX // 32, 0.01))
        logits = oq8.gemm(h, codes, scales)
        assert over.argmax_lowest(logits)[0] == 389
        packed = pack_q8(lb, codes, scales, N)
        call = lb.lowbit_draft_argmax_q8
    ws = Guarded((lb.lmhead_workspace_bytes(2, N, K_MAX),), torch.uint8, fill=0)
    out = Guarded((M,), torch.int32, fill=-1)
    call(bf16_dev(h), packed, M, N, K_MAX, dev(ids), out.t, ws.t)
    torch.cuda.synchronize()
    got = out.t.cpu().numpy()
    assert np.isin(got, ids).all()
    rows = np.searchsorted(ids, got)
    check_argmax(rows, logits, f"{fmt} draft K=65536 M={M}")
    assert not ws.t.any()
    ws.check(f"{fmt} draft workspace")
    out.check(f"{fmt} draft ids")
