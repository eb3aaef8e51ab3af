"""CPU checks of the C ABI: the library loads, exports every function include/lowbit.h
declares, and its host-only size/status queries behave as documented.  No kernel runs."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lowbit.h")


@pytest.fixture(scope="module")
def lib():
    from bit_weight_gemv_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted({n for n in names if n not in ("if", "defined")})


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("lowbit_pack_int4", "lowbit_pack_binplane", "lowbit_gemm_int4",
              "lowbit_gemm_binplane", "lmhead_argmax_verify"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_sizes_and_status_strings(lib):
    lib.lowbit_int4_packed_bytes.restype = ctypes.c_size_t
    lib.lowbit_binplane_packed_bytes.restype = ctypes.c_size_t
    lib.lmhead_workspace_bytes.restype = ctypes.c_size_t
    lib.lowbit_status_string.restype = ctypes.c_char_p
    # one 4B-class layer's INT4 projections: 50,012,160 payload bytes + 7 headers
    shapes = [(2560, 4096), (2560, 1024), (2560, 1024), (2560, 2560), (2560, 9728),
              (2560, 9728), (9728, 2560)]
    total = sum(lib.lowbit_int4_packed_bytes(n, k) - 128 for k, n in shapes)
    assert total == 50_012_160
    assert lib.lowbit_int4_packed_bytes(248_320, 4096) - 128 == 524_451_840
    assert lib.lowbit_int4_packed_bytes(32_768, 4096) - 128 == 69_206_016
    assert lib.lowbit_binplane_packed_bytes(3, 12288, 4096) - 128 == 21_233_664
    assert lib.lowbit_binplane_packed_bytes(4, 4096, 12288) - 128 == 28_311_552
    # ragged rows are padded to the 128-row tile
    assert lib.lowbit_int4_packed_bytes(33, 128) == 128 + 8448   # one 128-row tile, one group
    assert lib.lowbit_int4_packed_bytes(10, 100) == 0          # K not a multiple of 128
    assert lib.lowbit_binplane_packed_bytes(9, 32, 128) == 0   # P > 8
    assert lib.lmhead_workspace_bytes(16, 248_320, 4096) == 512
    assert lib.lmhead_workspace_bytes(1, 10, 128) == 0
    for s in range(7):
        assert lib.lowbit_status_string(s)
    assert lib.lowbit_status_string(0) == b"ok"


def test_host_validation_rejects_before_any_launch(lib):
    # Null pointers and bad shapes are rejected on the host; nothing reaches the GPU.
    vp = ctypes.c_void_p
    f = lib.lowbit_gemm_int4
    f.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
    assert f(None, None, 1, 64, 128, None, None) == 1            # invalid argument
    fake = vp(0x1000)
    assert f(fake, fake, 1, 64, 100, fake, None) == 2            # K % 128
    assert f(fake, fake, 33, 64, 128, fake, None) == 2           # M > 32
    assert f(vp(0x1008), fake, 1, 64, 128, fake, None) == 3      # X misaligned
    g = lib.lmhead_argmax_verify
    g.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp,
                  ctypes.c_size_t, vp]
    assert g(fake, fake, 16, 64, 128, fake, fake, fake, fake, fake, 100, None) == 4  # workspace
    assert g(fake, fake, 1, 64, 128, fake, fake, fake, fake, fake, 512, None) == 2   # M < 2


def test_kernel_family_selection_is_validated_on_the_host(lib):
    """The `_path` calls reject unknown families and shapes a family cannot take before
    touching the device (status 1 = invalid argument, 2 = shape)."""
    vp, ci = ctypes.c_void_p, ctypes.c_int
    fake = vp(0x1000)
    f = lib.lowbit_gemm_int4_path
    f.argtypes = [vp, vp, ci, ci, ci, vp, ci, vp]
    assert f(fake, fake, 16, 64, 128, fake, 4, None) == 1
    assert f(fake, fake, 16, 64, 128, fake, -1, None) == 1
    b = lib.lowbit_gemm_binplane_path
    b.argtypes = [vp, vp, ci, ci, ci, ci, vp, ci, vp]
    assert b(fake, fake, 3, 16, 64, 128, fake, 4, None) == 1
    sa = lib.lowbit_gemm_sa_path
    sa.argtypes = [vp, vp, ci, ci, ci, ci, ci, vp, ci, vp]
    assert sa(fake, fake, 3, 64, 16, 64, 256, fake, 4, None) == 1
    nv = lib.lowbit_gemm_nvfp4_path
    nv.argtypes = [vp, vp, ci, ci, ci, vp, ci, vp]
    assert nv(fake, fake, 2, 64, 128, fake, 1, None) == 2         # the streaming kernel is M = 1
    assert nv(fake, fake, 1, 64, 128, fake, 3, None) == 1
    d = lib.lowbit_draft_argmax_path
    d.argtypes = [vp, vp, ci, ci, ci, vp, vp, vp, ctypes.c_size_t, ci, vp]
    assert d(fake, fake, 2, 64, 128, None, fake, fake, 512, 1, None) == 2
    assert d(fake, fake, 1, 64, 128, None, fake, fake, 512, 7, None) == 1

    class Desc(ctypes.Structure):
        _fields_ = [("X", vp), ("packed", vp), ("Y", vp), ("N", ci), ("K", ci)]

    arr = (Desc * 2)(Desc(fake, fake, fake, 64, 128), Desc(fake, fake, fake, 32, 256))
    g = lib.lowbit_gemm_int4_grouped_path
    g.argtypes = [vp, ci, ci, ci, vp]
    assert g(ctypes.cast(arr, vp), 2, 16, 4, None) == 1
    assert g(ctypes.cast(arr, vp), 2, 5, 1, None) == 2           # the streaming kernel takes M <= 4
    assert g(ctypes.cast(arr, vp), 9, 16, 0, None) == 1           # at most 8 problems



def test_binding_refuses_host_tensors_and_empty_scalar_outputs(lib):
    """The Python binding passes raw pointers only for contiguous CUDA tensors of the declared
    dtype: host tensors are refused before anything reaches the library (there is no CPU
    path), and the one-element outputs of the verify calls must exist."""
    torch = pytest.importorskip("torch")
    import bit_weight_gemv_gb300 as lb
    from bit_weight_gemv_gb300 import _native
    X = torch.zeros((1, 128), dtype=torch.bfloat16)
    packed = torch.zeros(lb.lowbit_int4_packed_bytes(128, 128), dtype=torch.uint8)
    Y = torch.zeros((1, 128), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        lb.lowbit_gemm_int4(X, packed, 1, 128, 128, Y)
    with pytest.raises(TypeError):
        lb.lmhead_argmax_verify(X, packed, 1, 128, 128, torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, dtype=torch.int32),
                                torch.zeros(1, dtype=torch.int32), torch.zeros(512, dtype=torch.uint8))
    one, none = torch.zeros(1, dtype=torch.int32), torch.zeros(0, dtype=torch.int32)
    _native._need_scalar_outs(one, one)
    for a, b in ((none, one), (one, none)):
        with pytest.raises(ValueError):
            _native._need_scalar_outs(a, b)
