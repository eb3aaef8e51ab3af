"""GPU checks of lmhead_argmax_verify_noalloc, the LM-head verify step that uses the library's
own per-device scratch instead of a caller workspace (for callers that own no device
allocator).

The file is named to be collected last: the scratch is library state shared by every call on
the device, and these checks must hold whether they run alone in a fresh process or after all
other tests.  Each case makes two calls in a row and grades both against the oracle (argmax
where the oracle's top-1 margin exceeds 1e-2, acceptance bit-exact by the prefix rule on the
call's own argmax) and against lmhead_argmax_verify on the same inputs with a freshly zeroed
workspace, which runs the same kernel and so must agree exactly."""
import numpy as np
import pytest

import synth
from oracle import int4 as oint4
from oracle import verify as over
from helpers import bf16_dev, check_argmax, dev, f16_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_gemv_gb300 as lb
    return lb


def _outs(M):
    a = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    b = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    return a, n, b


@pytest.mark.parametrize("M,N,K,j", [(16, 1000, 512, None), (16, 32768, 4096, 15),
                                     (16, 32768, 4096, 0), (2, 40, 128, None), (32, 257, 256, 9)])
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls(lb, M, N, K, j):
    codes, scales, h = synth.int4_problem(21, M, N, K)
    logits = oint4.gemm(h, codes, scales)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), N, K, packed)
    drafts, planted = synth.plant_drafts(5, over.argmax_lowest(logits), N, j)
    H, D = bf16_dev(h), dev(drafts.astype(np.int32))
    margins = over.top2_margin(logits)

    ws = torch.zeros(lb.lmhead_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    a_ref, n_ref, b_ref = _outs(M)
    lb.lmhead_argmax_verify(H, packed, M, N, K, D, a_ref, n_ref, b_ref, ws)
    torch.cuda.synchronize()
    a_ref, n_ref, b_ref = a_ref.cpu().numpy(), int(n_ref.item()), int(b_ref.item())

    for call in range(2):
        a, n, b = _outs(M)
        lb.lmhead_argmax_verify_noalloc(H, packed, M, N, K, D, a, n, b)
        torch.cuda.synchronize()
        a = a.cpu().numpy()
        n, b = int(n.item()), int(b.item())
        check_argmax(a, logits, f"noalloc call {call}")
        assert (n, b) == over.accept(a, drafts), f"call {call}"
        if np.all(margins[:planted + 1] > 1e-2):
            assert n == planted, f"call {call}"
        # same kernel and rounding as the workspace entry point
        assert np.array_equal(a, a_ref), f"call {call}"
        assert (n, b) == (n_ref, b_ref), f"call {call}"
    assert lb.lowbit_device_error() == 0


def test_noalloc_rejects_bad_arguments_before_launch(lb):
    codes, scales, h = synth.int4_problem(0, 2, 64, 128)
    packed = torch.empty(lb.lowbit_int4_packed_bytes(64, 128), dtype=torch.uint8, device="cuda")
    lb.lowbit_pack_int4(dev(codes), f16_dev(scales), 64, 128, packed)
    H = torch.zeros((33, 128), dtype=torch.bfloat16, device="cuda")
    H[:2] = bf16_dev(h)
    D = dev(np.zeros(32, dtype=np.int32))
    a, n, b = _outs(33)
    for M, K, status in ((1, 128, 2), (33, 128, 2), (2, 100, 2)):
        with pytest.raises(lb.LowbitError) as e:
            lb.lmhead_argmax_verify_noalloc(H, packed, M, 64, K, D, a, n, b)
        assert e.value.status == status
    torch.cuda.synchronize()
    assert int(n.item()) == -1  # nothing was launched
