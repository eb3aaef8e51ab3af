"""ctypes marshalling for liblowbit.so (see the package docstring)."""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblowbit.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m bit_weight_gemv_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_SIGS = {
    "lowbit_status_string": (ctypes.c_char_p, [_i]),
    "lowbit_version": (_i, []),
    "lowbit_int4_packed_bytes": (_sz, [_i, _i]),
    "lowbit_binplane_packed_bytes": (_sz, [_i, _i, _i]),
    "lmhead_workspace_bytes": (_sz, [_i, _i, _i]),
    "lowbit_pack_int4": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "lowbit_pack_binplane": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "lowbit_validate_packed": (_i, [_vp, _i, _i, _i, _i, _vp]),
    "lowbit_gemm_int4": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "lowbit_gemm_binplane": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "lmhead_argmax_verify": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "lowbit_gemm_int4_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _i, _vp]),
    "lowbit_gemm_binplane_path": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _i, _vp]),
    "lmhead_argmax_verify_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _i, _vp]),
    "lowbit_device_error": (_i, [_vp, ctypes.POINTER(_i)]),
    "lowbit_debug_inject_stall": (_i, [_i]),
    "lmhead_argmax_partial": (_i, [_vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "lowbit_q8_packed_bytes": (_sz, [_i, _i]),
    "lowbit_pack_q8": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "lowbit_gemm_q8": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "lowbit_gemm_q8_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _i, _vp]),
    "lowbit_draft_argmax_q8": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "lmhead_accept_keys": (_i, [_vp, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "lowbit_sa_packed_bytes": (_sz, [_i, _i, _i, _i]),
    "lowbit_pack_sa": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp]),
    "lowbit_gemm_sa": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "lowbit_gemm_sa_path": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "lowbit_nvfp4_packed_bytes": (_sz, [_i, _i]),
    "lowbit_pack_nvfp4": (_i, [_vp, _vp, ctypes.c_float, _i, _i, _vp, _vp]),
    "lowbit_gemm_nvfp4": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "lowbit_gemm_nvfp4_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _i, _vp]),
    "lowbit_gemm_int4_grouped_path": (_i, [_vp, _i, _i, _i, _vp]),
    "lowbit_draft_argmax": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "lowbit_draft_argmax_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _sz, _i, _vp]),
}


class lowbit_gemm_desc(ctypes.Structure):
    """One multiply of lowbit_gemm_int4_grouped (mirrors the C struct)."""
    _fields_ = [("X", _vp), ("packed", _vp), ("Y", _vp), ("N", _i), ("K", _i)]


_SIGS["lowbit_gemm_int4_grouped"] = (_i, [ctypes.POINTER(lowbit_gemm_desc), _i, _i, _vp])
_SIGS["lmhead_argmax_verify_noalloc"] = (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp])
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class LowbitError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {lowbit_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise LowbitError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")


def _need_scalar_outs(n_accept, bonus):
    """The accepted count and the bonus token are written as one int32 each."""
    if n_accept.numel() < 1 or bonus.numel() < 1:
        raise ValueError("n_accept and bonus must hold one element each")


def lowbit_status_string(status: int) -> str:
    return lib.lowbit_status_string(int(status)).decode()


def lowbit_version() -> int:
    return lib.lowbit_version()


def lowbit_int4_packed_bytes(N: int, K: int) -> int:
    return lib.lowbit_int4_packed_bytes(N, K)


def lowbit_binplane_packed_bytes(P: int, N: int, K: int) -> int:
    return lib.lowbit_binplane_packed_bytes(P, N, K)


def lmhead_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib.lmhead_workspace_bytes(M, N, K)


def lowbit_pack_int4(codes, scales, N, K, packed, stream=None):
    """codes int8 [N][K], scales fp16 [N][K/128] -> packed uint8 [lowbit_int4_packed_bytes]."""
    _need(codes, torch.int8, "codes")
    _need(scales, torch.float16, "scales")
    _need(packed, torch.uint8, "packed")
    if packed.numel() < lowbit_int4_packed_bytes(N, K):
        raise ValueError("packed buffer too small")
    _check(lib.lowbit_pack_int4(_ptr(codes), _ptr(scales), N, K, _ptr(packed), _stream(stream)),
           "lowbit_pack_int4")


def lowbit_pack_binplane(signbits, alpha, P, N, K, packed, stream=None):
    """signbits uint8 [P][N][K/8], alpha fp16 [P][N][K/128] -> packed uint8."""
    _need(signbits, torch.uint8, "signbits")
    _need(alpha, torch.float16, "alpha")
    _need(packed, torch.uint8, "packed")
    if packed.numel() < lowbit_binplane_packed_bytes(P, N, K):
        raise ValueError("packed buffer too small")
    _check(lib.lowbit_pack_binplane(_ptr(signbits), _ptr(alpha), P, N, K, _ptr(packed),
                                    _stream(stream)), "lowbit_pack_binplane")


def lowbit_validate_packed(packed, fmt, P, N, K, stream=None) -> int:
    """Synchronous header check; returns the status code (0 = matches)."""
    _need(packed, torch.uint8, "packed")
    return lib.lowbit_validate_packed(_ptr(packed), fmt, P, N, K, _stream(stream))


def _gemm_args(X, packed, M, N, K, Y):
    _need(X, torch.bfloat16, "X")
    _need(packed, torch.uint8, "packed")
    _need(Y, torch.bfloat16, "Y")
    if X.numel() < M * K or Y.numel() < M * N:
        raise ValueError("X or Y too small")


def lowbit_gemm_int4(X, packed, M, N, K, Y, stream=None):
    """Y bf16 [M][N] = X bf16 [M][K] times the packed INT4 weights, transposed."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_int4(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), _stream(stream)),
           "lowbit_gemm_int4")


def lowbit_gemm_int4_path(X, packed, M, N, K, Y, path, stream=None):
    """lowbit_gemm_int4 with the kernel family forced (1 = CUDA cores, 2 = tcgen05, 3 = warp MMA)."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_int4_path(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), path,
                                     _stream(stream)), "lowbit_gemm_int4_path")


def _descs(problems, M):
    n = len(problems)
    arr = (lowbit_gemm_desc * max(1, n))()
    for i, (X, packed, N, K, Y) in enumerate(problems):
        _gemm_args(X, packed, M, N, K, Y)
        arr[i] = lowbit_gemm_desc(X.data_ptr(), packed.data_ptr(), Y.data_ptr(), N, K)
    return arr, n


def lowbit_gemm_int4_grouped(problems, M, stream=None):
    """Several independent INT4 multiplies with a common M in one call.

    problems: sequence of (X, packed, N, K, Y) tuples, 1 to 8 of them."""
    arr, n = _descs(problems, M)
    _check(lib.lowbit_gemm_int4_grouped(arr, n, M, _stream(stream)), "lowbit_gemm_int4_grouped")


def lowbit_gemm_int4_grouped_path(problems, M, path, stream=None):
    """lowbit_gemm_int4_grouped with the kernel family forced (1 = streaming, M <= 4;
    2 = tcgen05; 3 = warp-level MMA)."""
    arr, n = _descs(problems, M)
    _check(lib.lowbit_gemm_int4_grouped_path(arr, n, M, path, _stream(stream)),
           "lowbit_gemm_int4_grouped_path")


def lowbit_gemm_binplane(X, packed, P, M, N, K, Y, stream=None):
    """Y bf16 [M][N] = X bf16 [M][K] times the packed binary-plane weights, transposed."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_binplane(_ptr(X), _ptr(packed), P, M, N, K, _ptr(Y), _stream(stream)),
           "lowbit_gemm_binplane")


def lowbit_gemm_binplane_path(X, packed, P, M, N, K, Y, path, stream=None):
    """lowbit_gemm_binplane with the kernel family forced (1 = CUDA cores, 2 = tcgen05, 3 = warp MMA)."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_binplane_path(_ptr(X), _ptr(packed), P, M, N, K, _ptr(Y), path,
                                         _stream(stream)), "lowbit_gemm_binplane_path")


def lowbit_sa_packed_bytes(P: int, G: int, N: int, K: int) -> int:
    return lib.lowbit_sa_packed_bytes(P, G, N, K)


def lowbit_pack_sa(signbits, codes, d, P, G, N, K, packed, stream=None):
    """signbits uint8 [P][N][K/8], codes uint8 [P][N][K/G], d fp16 [N][K/256] -> packed uint8."""
    _need(signbits, torch.uint8, "signbits")
    _need(codes, torch.uint8, "codes")
    _need(d, torch.float16, "d")
    _need(packed, torch.uint8, "packed")
    if packed.numel() < lowbit_sa_packed_bytes(P, G, N, K):
        raise ValueError("packed buffer too small")
    _check(lib.lowbit_pack_sa(_ptr(signbits), _ptr(codes), _ptr(d), P, G, N, K, _ptr(packed),
                              _stream(stream)), "lowbit_pack_sa")


def lowbit_gemm_sa(X, packed, P, G, M, N, K, Y, stream=None):
    """Y bf16 [M][N] = X bf16 [M][K] times the packed sa-format weights, transposed."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_sa(_ptr(X), _ptr(packed), P, G, M, N, K, _ptr(Y), _stream(stream)),
           "lowbit_gemm_sa")


def lowbit_gemm_sa_path(X, packed, P, G, M, N, K, Y, path, stream=None):
    """lowbit_gemm_sa with the kernel family forced (1 = CUDA cores, 2 = tcgen05, 3 = warp MMA)."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_sa_path(_ptr(X), _ptr(packed), P, G, M, N, K, _ptr(Y), path,
                                   _stream(stream)), "lowbit_gemm_sa_path")


def lowbit_nvfp4_packed_bytes(N: int, K: int) -> int:
    return lib.lowbit_nvfp4_packed_bytes(N, K)


def lowbit_pack_nvfp4(codes, scales, g, N, K, packed, stream=None):
    """codes uint8 [N][K/2] (E2M1 pairs), scales uint8 [N][K/16] (E4M3), g float -> packed."""
    _need(codes, torch.uint8, "codes")
    _need(scales, torch.uint8, "scales")
    _need(packed, torch.uint8, "packed")
    if packed.numel() < lowbit_nvfp4_packed_bytes(N, K):
        raise ValueError("packed buffer too small")
    _check(lib.lowbit_pack_nvfp4(_ptr(codes), _ptr(scales), float(g), N, K, _ptr(packed),
                                 _stream(stream)), "lowbit_pack_nvfp4")


def lowbit_gemm_nvfp4(X, packed, M, N, K, Y, stream=None):
    """Y bf16 [M][N] = X bf16 [M][K] times the packed NVFP4 weights, transposed."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_nvfp4(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), _stream(stream)),
           "lowbit_gemm_nvfp4")


def lowbit_gemm_nvfp4_path(X, packed, M, N, K, Y, path, stream=None):
    """lowbit_gemm_nvfp4 with the kernel forced (1 = streaming mat-vec, M = 1; 2 = tensor cores)."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_nvfp4_path(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), path,
                                      _stream(stream)), "lowbit_gemm_nvfp4_path")


def _draft_args(H, packed_head, M, N, K, id_map, ids, workspace):
    _need(H, torch.bfloat16, "H")
    _need(packed_head, torch.uint8, "packed_head")
    _need(ids, torch.int32, "ids")
    _need(workspace, torch.uint8, "workspace")
    if id_map is not None:
        _need(id_map, torch.int32, "id_map")
        if id_map.numel() < N:
            raise ValueError("id_map too small")
    if H.numel() < M * K or ids.numel() < M:
        raise ValueError("H or ids too small")


def lowbit_draft_argmax(H, packed_head, M, N, K, id_map, ids, workspace, stream=None):
    """ids int32 [M] = id_map[argmax over the N rows of an NVFP4 draft head] (id_map may be None)."""
    _draft_args(H, packed_head, M, N, K, id_map, ids, workspace)
    _check(lib.lowbit_draft_argmax(_ptr(H), _ptr(packed_head), M, N, K, _ptr(id_map), _ptr(ids),
                                   _ptr(workspace), workspace.numel(), _stream(stream)),
           "lowbit_draft_argmax")


def lowbit_draft_argmax_path(H, packed_head, M, N, K, id_map, ids, workspace, path, stream=None):
    """lowbit_draft_argmax with the kernel forced (1 = streaming mat-vec, M = 1; 2 = tensor cores)."""
    _draft_args(H, packed_head, M, N, K, id_map, ids, workspace)
    _check(lib.lowbit_draft_argmax_path(_ptr(H), _ptr(packed_head), M, N, K, _ptr(id_map),
                                        _ptr(ids), _ptr(workspace), workspace.numel(), path,
                                        _stream(stream)), "lowbit_draft_argmax_path")


def _lmhead_args(H, packed_head, M, K, draft, argmax, n_accept, bonus, workspace):
    _need(H, torch.bfloat16, "H")
    _need(packed_head, torch.uint8, "packed_head")
    for t, nm in ((draft, "draft"), (argmax, "argmax"), (n_accept, "n_accept"), (bonus, "bonus")):
        _need(t, torch.int32, nm)
    _need(workspace, torch.uint8, "workspace")
    if H.numel() < M * K or draft.numel() < M - 1 or argmax.numel() < M:
        raise ValueError("H, draft or argmax too small")
    _need_scalar_outs(n_accept, bonus)


def lmhead_argmax_verify(H, packed_head, M, N, K, draft, argmax, n_accept, bonus, workspace,
                         stream=None):
    """Fused LM-head argmax over N vocabulary rows plus greedy prefix acceptance."""
    _lmhead_args(H, packed_head, M, K, draft, argmax, n_accept, bonus, workspace)
    _check(lib.lmhead_argmax_verify(_ptr(H), _ptr(packed_head), M, N, K, _ptr(draft), _ptr(argmax),
                                    _ptr(n_accept), _ptr(bonus), _ptr(workspace),
                                    workspace.numel(), _stream(stream)), "lmhead_argmax_verify")


def lmhead_argmax_verify_path(H, packed_head, M, N, K, draft, argmax, n_accept, bonus, workspace,
                              path, stream=None):
    """lmhead_argmax_verify with the kernel family forced (1 = CUDA cores, 2 = tcgen05, 3 = warp MMA)."""
    _lmhead_args(H, packed_head, M, K, draft, argmax, n_accept, bonus, workspace)
    _check(lib.lmhead_argmax_verify_path(_ptr(H), _ptr(packed_head), M, N, K, _ptr(draft),
                                         _ptr(argmax), _ptr(n_accept), _ptr(bonus),
                                         _ptr(workspace), workspace.numel(), path,
                                         _stream(stream)), "lmhead_argmax_verify_path")


def lmhead_argmax_verify_noalloc(H, packed_head, M, N, K, draft, argmax, n_accept, bonus,
                                 stream=None):
    """lmhead_argmax_verify using the library's per-device scratch instead of a workspace
    (for callers that cannot allocate; concurrent calls on one device race)."""
    _need(H, torch.bfloat16, "H")
    _need(packed_head, torch.uint8, "packed_head")
    for t, nm in ((draft, "draft"), (argmax, "argmax"), (n_accept, "n_accept"), (bonus, "bonus")):
        _need(t, torch.int32, nm)
    if H.numel() < M * K or draft.numel() < M - 1 or argmax.numel() < M:
        raise ValueError("H, draft or argmax too small")
    _need_scalar_outs(n_accept, bonus)
    _check(lib.lmhead_argmax_verify_noalloc(_ptr(H), _ptr(packed_head), M, N, K, _ptr(draft),
                                            _ptr(argmax), _ptr(n_accept), _ptr(bonus),
                                            _stream(stream)), "lmhead_argmax_verify_noalloc")


def lowbit_device_error(stream=None) -> int:
    """Synchronise and return (then clear) the device's recorded kernel-side error."""
    out = ctypes.c_int(0)
    _check(lib.lowbit_device_error(_stream(stream), ctypes.byref(out)), "lowbit_device_error")
    return out.value


def lowbit_debug_inject_stall(on: bool) -> None:
    """Testing only: make later streaming / warp-MMA launches give up on their data waits."""
    _check(lib.lowbit_debug_inject_stall(1 if on else 0), "lowbit_debug_inject_stall")


def lmhead_argmax_partial(H, packed_shard, M, N, K, row_offset, keys_out, workspace, stream=None):
    """One shard of a row-sharded LM head: keys_out int64 [M] = the slice's best
    (logit, global row) key per token (see include/lowbit.h)."""
    _need(H, torch.bfloat16, "H")
    _need(packed_shard, torch.uint8, "packed_shard")
    _need(keys_out, torch.int64, "keys_out")
    _need(workspace, torch.uint8, "workspace")
    if H.numel() < M * K or keys_out.numel() < M:
        raise ValueError("H or keys_out too small")
    _check(lib.lmhead_argmax_partial(_ptr(H), _ptr(packed_shard), M, N, K, row_offset,
                                     _ptr(keys_out), _ptr(workspace), workspace.numel(),
                                     _stream(stream)), "lmhead_argmax_partial")


def lmhead_accept_keys(keys, W, M, draft, argmax, n_accept, bonus, stream=None):
    """Merge W shards' keys (int64 [W][M]) into the full head's argmax, then greedy acceptance."""
    _need(keys, torch.int64, "keys")
    for t, nm in ((draft, "draft"), (argmax, "argmax"), (n_accept, "n_accept"), (bonus, "bonus")):
        _need(t, torch.int32, nm)
    if keys.numel() < W * M or draft.numel() < M - 1 or argmax.numel() < M:
        raise ValueError("keys, draft or argmax too small")
    _need_scalar_outs(n_accept, bonus)
    _check(lib.lmhead_accept_keys(_ptr(keys), W, M, _ptr(draft), _ptr(argmax), _ptr(n_accept),
                                  _ptr(bonus), _stream(stream)), "lmhead_accept_keys")


def lowbit_q8_packed_bytes(N: int, K: int) -> int:
    return lib.lowbit_q8_packed_bytes(N, K)


def lowbit_pack_q8(codes, scales, N, K, packed, stream=None):
    """codes int8 [N][K], scales fp16 [N][K/32] -> packed uint8 [lowbit_q8_packed_bytes]."""
    _need(codes, torch.int8, "codes")
    _need(scales, torch.float16, "scales")
    _need(packed, torch.uint8, "packed")
    if packed.numel() < lowbit_q8_packed_bytes(N, K):
        raise ValueError("packed buffer too small")
    _check(lib.lowbit_pack_q8(_ptr(codes), _ptr(scales), N, K, _ptr(packed), _stream(stream)),
           "lowbit_pack_q8")


def lowbit_gemm_q8(X, packed, M, N, K, Y, stream=None):
    """Y bf16 [M][N] = X bf16 [M][K] times the packed Q8 weights, transposed."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_q8(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), _stream(stream)),
           "lowbit_gemm_q8")


def lowbit_gemm_q8_path(X, packed, M, N, K, Y, path, stream=None):
    """lowbit_gemm_q8 with the kernel forced (1 = streaming, M = 1; 3 = warp-level MMA)."""
    _gemm_args(X, packed, M, N, K, Y)
    _check(lib.lowbit_gemm_q8_path(_ptr(X), _ptr(packed), M, N, K, _ptr(Y), path, _stream(stream)),
           "lowbit_gemm_q8_path")


def lowbit_draft_argmax_q8(H, packed_head, M, N, K, id_map, ids, workspace, stream=None):
    """ids int32 [M] = id_map[argmax over the N rows of a Q8 draft head] (id_map may be None)."""
    _draft_args(H, packed_head, M, N, K, id_map, ids, workspace)
    _check(lib.lowbit_draft_argmax_q8(_ptr(H), _ptr(packed_head), M, N, K, _ptr(id_map), _ptr(ids),
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "lowbit_draft_argmax_q8")
