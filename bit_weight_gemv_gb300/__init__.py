"""Python binding of liblowbit.so: low-bit weight GEMV/GEMM for speculative decoding on GB300.

Argument marshalling only: every function takes torch tensors (device memory owned by the
caller), checks dtypes/shapes, passes raw pointers and the current CUDA stream to the C ABI
(include/lowbit.h) under the same name, and raises LowbitError on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU fallback.  The in-tree
liblowbit.so is loaded on first use of any of these names and its absence raises
ImportError (build it with ``python -m bit_weight_gemv_gb300.build``).
"""

__all__ = [
    "LIB_PATH", "LowbitError", "lib", "lmhead_argmax_verify", "lmhead_workspace_bytes",
    "lowbit_binplane_packed_bytes", "lowbit_device_error", "lowbit_gemm_binplane",
    "lowbit_gemm_int4", "lowbit_int4_packed_bytes", "lowbit_pack_binplane", "lowbit_pack_int4",
    "lowbit_status_string", "lowbit_validate_packed", "lowbit_version",
    "lowbit_gemm_int4_path", "lowbit_gemm_binplane_path", "lmhead_argmax_verify_path",
    "lowbit_gemm_int4_grouped", "lowbit_gemm_int4_grouped_path", "lowbit_gemm_desc", "lmhead_argmax_verify_noalloc",
    "lowbit_sa_packed_bytes", "lowbit_pack_sa", "lowbit_gemm_sa", "lowbit_gemm_sa_path",
    "lowbit_nvfp4_packed_bytes", "lowbit_pack_nvfp4", "lowbit_gemm_nvfp4", "lowbit_gemm_nvfp4_path",
    "lowbit_draft_argmax", "lowbit_draft_argmax_path",
    "lowbit_debug_inject_stall",
    "lmhead_argmax_partial", "lmhead_accept_keys",
    "lowbit_q8_packed_bytes", "lowbit_pack_q8", "lowbit_gemm_q8", "lowbit_gemm_q8_path",
    "lowbit_draft_argmax_q8",
]


def __getattr__(name):
    if name in __all__:
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)
