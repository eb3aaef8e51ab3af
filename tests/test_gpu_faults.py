"""GPU checks of the bounded waits' give-up path, and canary bands around outputs.

The library's test-only stall setting (lowbit_debug_inject_stall) makes the compute warps of
the streaming and warp-MMA kernels wait for their data on an mbarrier that nothing arrives on
(a flag nothing sets), with a short limit; no memory is touched out of bounds and no GPU fault
is involved.  Every such call must record LOWBIT_ERR_TIMEOUT, write no output, leave the LM-head
workspace zeroed, and leave the context usable: the same call made normally afterwards matches
the oracle."""
import numpy as np
import pytest

import synth
from oracle import binplane as obp
from oracle import int4 as oint4
from oracle import nvfp4 as onf
from oracle import sa as osa
from oracle import verify as over
from helpers import Guarded, bf16_dev, check_argmax, check_gemm, dev, f16_dev, host_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TIMEOUT = 5


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    lb.lowbit_device_error()  # start from a clear error word
    return lb


def _stalled(lb, call):
    """Run `call` under the stall setting; return the recorded device error."""
    lb.lowbit_debug_inject_stall(True)
    try:
        call()
    finally:
        lb.lowbit_debug_inject_stall(False)
    return lb.lowbit_device_error()


def _pack_int4(lb, codes, scales):
    N, K = codes.shape
    p = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, p)
    return p


# (M, N, K): M=1 and 2 run the streaming kernel, 16 and 32 the warp-level MMA; K = 9728 splits
# each tile's groups over a cluster (the split-K exchange), N = 300 leaves a ragged tile.
@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (1, 2560, 9728), (2, 1024, 2560),
                                   (16, 300, 1024), (16, 2560, 9728), (32, 257, 2560)])
def test_int4_stall_times_out_writes_nothing_then_recovers(lb, M, N, K):
    codes, scales, x = synth.int4_problem(41, M, N, K)
    P, X = _pack_int4(lb, codes, scales), bf16_dev(x)
    Y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    before = host_bits(Y.t).copy()
    assert _stalled(lb, lambda: lb.lowbit_gemm_int4(X, P, M, N, K, Y.t)) == TIMEOUT
    assert np.array_equal(host_bits(Y.t), before), "a timed-out call wrote outputs"
    Y.check("stalled int4")
    lb.lowbit_gemm_int4(X, P, M, N, K, Y.t)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y.t), oint4.gemm(x, codes, scales), f"int4 after stall M={M}")
    Y.check("int4")
    assert lb.lowbit_device_error() == 0


def test_grouped_stall_times_out_and_recovers(lb):
    shapes = ((2560, 4096), (2560, 1024), (9728, 2560))
    probs, refs, outs = [], [], []
    for j, (K, N) in enumerate(shapes):
        codes, scales, x = synth.int4_problem(42, 1, N, K, j)
        Y = Guarded((1, N), torch.bfloat16, fill=float("nan"))
        probs.append((bf16_dev(x), _pack_int4(lb, codes, scales), N, K, Y.t))
        refs.append(oint4.gemm(x, codes, scales))
        outs.append(Y)
    assert _stalled(lb, lambda: lb.lowbit_gemm_int4_grouped(probs, 1)) == TIMEOUT
    for Y in outs:
        assert torch.isnan(Y.t.float()).all()
        Y.check("stalled grouped")
    lb.lowbit_gemm_int4_grouped(probs, 1)
    torch.cuda.synchronize()
    for j, (Y, r) in enumerate(zip(outs, refs)):
        check_gemm(host_bits(Y.t), r, f"grouped after stall {j}")
        Y.check("grouped")
    assert lb.lowbit_device_error() == 0


@pytest.mark.parametrize("M", [1, 16])
def test_binplane_and_sa_stall_times_out_and_recovers(lb, M):
    P, N, K = 3, 400, 1024
    bits, alpha, x = synth.binplane_problem(43, P, M, N, K)
    pk = torch.empty(lb.lowbit_binplane_packed_bytes(P, N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_binplane(dev(bits), f16_dev(alpha), P, N, K, pk)
    Y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    assert _stalled(lb, lambda: lb.lowbit_gemm_binplane(bf16_dev(x), pk, P, M, N, K, Y.t)) == TIMEOUT
    assert torch.isnan(Y.t.float()).all()
    Y.check("stalled binplane")
    lb.lowbit_gemm_binplane(bf16_dev(x), pk, P, M, N, K, Y.t)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y.t), obp.gemm(x, bits, alpha), f"binplane after stall M={M}")
    Y.check("binplane")

    G = 64
    bits, codes, d, x = synth.sa_problem(43, P, G, M, N, K)
    pk = torch.empty(lb.lowbit_sa_packed_bytes(P, G, N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_sa(dev(bits), dev(codes), f16_dev(d), P, G, N, K, pk)
    Y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    assert _stalled(lb, lambda: lb.lowbit_gemm_sa(bf16_dev(x), pk, P, G, M, N, K, Y.t)) == TIMEOUT
    assert torch.isnan(Y.t.float()).all()
    Y.check("stalled sa")
    lb.lowbit_gemm_sa(bf16_dev(x), pk, P, G, M, N, K, Y.t)
    torch.cuda.synchronize()
    check_gemm(host_bits(Y.t), osa.gemm(x, bits, codes, d, G), f"sa after stall M={M}")
    assert lb.lowbit_device_error() == 0


@pytest.mark.parametrize("N,K", [(2000, 512), (4096, 9728)])
def test_lmhead_stall_writes_nothing_and_resets_workspace(lb, N, K):
    M = 16
    codes, scales, h = synth.int4_problem(44, M, N, K)
    logits = oint4.gemm(h, codes, scales)
    drafts, _ = synth.plant_drafts(44, over.argmax_lowest(logits), N, 7)
    P, H, D = _pack_int4(lb, codes, scales), bf16_dev(h), dev(drafts)
    ws = Guarded((lb.lmhead_workspace_bytes(M, N, K),), torch.uint8, fill=0)
    a = Guarded((M,), torch.int32, fill=-7)
    n = Guarded((1,), torch.int32, fill=-7)
    b = Guarded((1,), torch.int32, fill=-7)
    call = lambda: lb.lmhead_argmax_verify(H, P, M, N, K, D, a.t, n.t, b.t, ws.t)
    assert _stalled(lb, call) == TIMEOUT
    assert (a.t == -7).all() and int(n.t.item()) == -7 and int(b.t.item()) == -7
    assert not ws.t.any(), "workspace not left zeroed"
    for g in (ws, a, n, b):
        g.check("stalled lmhead")
    call()
    torch.cuda.synchronize()
    got = a.t.cpu().numpy()
    check_argmax(got, logits, "lmhead after stall")
    assert (int(n.t.item()), int(b.t.item())) == over.accept(got, drafts)
    assert not ws.t.any()
    for g in (ws, a, n, b):
        g.check("lmhead")
    assert lb.lowbit_device_error() == 0


def test_draft_head_stall_writes_nothing_and_resets_workspace(lb):
    N, K = 4096, 2048
    codes, scales, g, ids, h = synth.nvfp4_problem(45, 1, N, K)
    pk = torch.empty(lb.lowbit_nvfp4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_nvfp4(dev(codes), dev(scales), g, N, K, pk)
    ws = Guarded((lb.lmhead_workspace_bytes(2, N, K),), torch.uint8, fill=0)
    out = Guarded((1,), torch.int32, fill=-7)
    idm = dev(ids)
    call = lambda: lb.lowbit_draft_argmax(bf16_dev(h), pk, 1, N, K, idm, out.t, ws.t)
    assert _stalled(lb, call) == TIMEOUT
    assert int(out.t.item()) == -7 and not ws.t.any()
    call()
    torch.cuda.synchronize()
    check_argmax(np.searchsorted(ids, out.t.cpu().numpy()), onf.gemm(h, codes, scales, g), "draft")
    for gd in (ws, out):
        gd.check("draft")
    assert lb.lowbit_device_error() == 0


@pytest.mark.parametrize("M", [1, 16])
def test_q8_stall_times_out_and_recovers(lb, M):
    from oracle import q8 as oq8
    N, K = 700, 2048
    codes, scales, ids, h = synth.q8_problem(46, M, N, K)
    pk = torch.empty(lb.lowbit_q8_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_q8(dev(codes), f16_dev(scales), N, K, pk)
    Y = Guarded((M, N), torch.bfloat16, fill=float("nan"))
    assert _stalled(lb, lambda: lb.lowbit_gemm_q8(bf16_dev(h), pk, M, N, K, Y.t)) == TIMEOUT
    assert torch.isnan(Y.t.float()).all()
    ws = Guarded((lb.lmhead_workspace_bytes(2, N, K),), torch.uint8, fill=0)
    out = Guarded((M,), torch.int32, fill=-7)
    call = lambda: lb.lowbit_draft_argmax_q8(bf16_dev(h), pk, M, N, K, dev(ids), out.t, ws.t)
    assert _stalled(lb, call) == TIMEOUT
    assert (out.t == -7).all() and not ws.t.any()
    lb.lowbit_gemm_q8(bf16_dev(h), pk, M, N, K, Y.t)
    call()
    torch.cuda.synchronize()
    logits = oq8.gemm(h, codes, scales)
    check_gemm(host_bits(Y.t), logits, f"q8 after stall M={M}")
    check_argmax(np.searchsorted(ids, out.t.cpu().numpy()), logits, "q8 draft after stall")
    for g in (Y, ws, out):
        g.check("q8 stall")
    assert lb.lowbit_device_error() == 0
