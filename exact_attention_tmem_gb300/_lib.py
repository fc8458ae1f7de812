"""ctypes binding of libfa_gb300.so (the C ABI in include/fa.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their data pointers and the current CUDA stream go through the C
ABI, and a non-zero status becomes an ``FaError``.  Every step of the
computation runs in the library's kernels; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ALIGNMENT = 3
FA_ERR_WORKSPACE = 4
FA_ERR_CUDA = 5
FA_ERR_DEVICE_TIMEOUT = 6

EXPORTED = ("fa_fwd", "fa_fwd_gqa", "fa_fwd_f32", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_gqa",
            "fa_bwd_deterministic_workspace_size", "fa_bwd_deterministic", "fa_bwd_noalloc",
            "fa_fwd_bwd_host_buffer_size", "fa_fwd_bwd_host",
            "fa_decode_workspace_size", "fa_decode",
            "fa_fp8_v_bytes", "fa_quantize_qk_fp8", "fa_quantize_v_fp8", "fa_fwd_fp8",
            "fa_get_device_status", "fa_selftest_wait_timeout", "fa_status_string",
            "fa_last_cuda_error")
NOALLOC_SCRATCH_BYTES = 64 << 20   # FA_NOALLOC_SCRATCH_BYTES in include/fa.h

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status}"
                         + (f", cudaError {last_cuda_error()})" if status == FA_ERR_CUDA else ")"))


def load() -> ctypes.CDLL:
    """Load the library (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "exact_attention_tmem_gb300.build.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, vp]
        lib.fa_fwd.restype = I
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, I, F, I, vp]
        lib.fa_fwd_gqa.restype = I
        lib.fa_fwd_f32.argtypes = [vp, vp, vp, vp, vp, I, I, I, I, F, I, vp]
        lib.fa_fwd_f32.restype = I
        lib.fa_bwd_workspace_size.argtypes = [I, I, I, I]
        lib.fa_bwd_workspace_size.restype = Z
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, Z, I, I, I, I, F, I, vp]
        lib.fa_bwd.restype = I
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, Z, I, I, I, I, I, F, I, vp]
        lib.fa_bwd_gqa.restype = I
        lib.fa_bwd_deterministic_workspace_size.argtypes = [I, I, I, I]
        lib.fa_bwd_deterministic_workspace_size.restype = Z
        lib.fa_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, Z, I, I, I, I, I, F, I, vp]
        lib.fa_bwd_deterministic.restype = I
        lib.fa_decode_workspace_size.argtypes = [I, I, I, I, I]
        lib.fa_decode_workspace_size.restype = Z
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, vp, Z, I, I, I, I, I, F, I, vp]
        lib.fa_decode.restype = I
        lib.fa_fp8_v_bytes.argtypes = [I, I, I, I]
        lib.fa_fp8_v_bytes.restype = Z
        lib.fa_quantize_qk_fp8.argtypes = [vp, vp, vp, vp, I, I, I, I, vp]
        lib.fa_quantize_qk_fp8.restype = I
        lib.fa_quantize_v_fp8.argtypes = [vp, vp, vp, I, I, I, I, vp]
        lib.fa_quantize_v_fp8.restype = I
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, I, F, I, vp]
        lib.fa_fwd_fp8.restype = I
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, I, I, I, I, F, I, vp]
        lib.fa_bwd_noalloc.restype = I
        lib.fa_fwd_bwd_host_buffer_size.argtypes = [I, I, I, I, I]
        lib.fa_fwd_bwd_host_buffer_size.restype = Z
        lib.fa_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, Z, I, I, I, I, F, I, I, vp]
        lib.fa_fwd_bwd_host.restype = I
        lib.fa_get_device_status.argtypes = [vp]
        lib.fa_get_device_status.restype = I
        lib.fa_selftest_wait_timeout.argtypes = [vp]
        lib.fa_selftest_wait_timeout.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_cuda_error.argtypes = []
        lib.fa_last_cuda_error.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def last_cuda_error() -> int:
    return int(load().fa_last_cuda_error())


def check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)
