"""The C-ABI library: it loads, exports every declared entry point, and rejects bad
arguments on the host with the documented status codes (no GPU needed)."""
import ctypes
import os
import re

import pytest

from exact_attention_tmem_gb300 import _lib
from exact_attention_tmem_gb300 import buildlib as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")

A = 0x10000   # fake, 16-byte aligned "device" addresses: never dereferenced on the host
W = 0x20000


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings(lib):
    for code in range(0, 7):
        s = _lib.status_string(code)
        assert s and s != "unknown status"
    assert _lib.status_string(99) == "unknown status"


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=128, scale=0.1, causal=0, f32=False):
    fn = lib.fa_fwd_f32 if f32 else lib.fa_fwd
    return fn(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, None)


def bwd(lib, ptrs=None, ws=W, ws_bytes=None, B=1, H=1, N=128, d=128, scale=0.1):
    p = [A] * 9 if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_workspace_size(B, H, N, d) if B > 0 and H > 0 and N > 0 else 0
    return lib.fa_bwd(*p, ws, ws_bytes, B, H, N, d, ctypes.c_float(scale), 1, None)


@pytest.mark.parametrize("which", range(5))
def test_fwd_null_pointer(lib, which):
    ptrs = [A] * 5
    ptrs[which] = None
    assert fwd(lib, *ptrs) == _lib.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("B,H,N", [(0, 1, 8), (1, 0, 8), (1, 1, 0), (-1, 1, 8), (1, 1, -5)])
def test_fwd_bad_sizes(lib, B, H, N):
    assert fwd(lib, B=B, H=H, N=N) == _lib.FA_ERR_INVALID_ARG


def test_fwd_size_overflow(lib):
    # B*H above INT_MAX, and B*H*N*d above 2^62
    assert fwd(lib, B=1 << 20, H=1 << 20, N=8) == _lib.FA_ERR_INVALID_ARG
    assert fwd(lib, B=1 << 15, H=1 << 15, N=(1 << 31) - 1) == _lib.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), float("-inf")])
def test_fwd_non_finite_scale(lib, scale):
    assert fwd(lib, scale=scale) == _lib.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [1, 32, 96, 256])
def test_fwd_unsupported_head_dim(lib, d):
    assert fwd(lib, d=d) == _lib.FA_ERR_UNSUPPORTED


def test_fwd_f32_only_d64(lib):
    assert fwd(lib, d=128, f32=True) == _lib.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("which,addr", [(0, A + 8), (1, A + 2), (2, A + 4), (3, A + 1), (4, A + 2)])
def test_fwd_misaligned(lib, which, addr):
    ptrs = [A] * 5
    ptrs[which] = addr
    assert fwd(lib, *ptrs) == _lib.FA_ERR_ALIGNMENT


def test_fwd_lse_needs_only_4_byte_alignment(lib):
    # lse at A+4 passes the host checks; what follows needs a device
    st = fwd(lib, lse=A + 4)
    assert st in (_lib.FA_ERR_CUDA, _lib.FA_ERR_UNSUPPORTED) or st == _lib.FA_OK


def test_workspace_size(lib):
    B, H, N, d = 2, 3, 300, 64
    npad = 384
    acc = B * H * N * d * 4
    vec = -(-(B * H * npad * 4) // 256) * 256
    assert lib.fa_bwd_workspace_size(B, H, N, d) == -(-acc // 256) * 256 + 2 * vec
    assert lib.fa_bwd_workspace_size(0, 1, 8, 64) == 0
    assert lib.fa_bwd_workspace_size(1, 1, 8, 96) == 0


@pytest.mark.parametrize("which", range(9))
def test_bwd_null_pointer(lib, which):
    ptrs = [A] * 9
    ptrs[which] = None
    assert bwd(lib, ptrs) == _lib.FA_ERR_INVALID_ARG


def test_bwd_workspace_checks(lib):
    assert bwd(lib, ws=None) == _lib.FA_ERR_WORKSPACE
    need = lib.fa_bwd_workspace_size(1, 1, 128, 128)
    assert bwd(lib, ws_bytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert bwd(lib, ws=W + 16) == _lib.FA_ERR_ALIGNMENT


@pytest.mark.parametrize("which", [0, 1, 2, 3, 5, 6, 7, 8])
def test_bwd_misaligned(lib, which):
    ptrs = [A] * 9
    ptrs[which] = A + 8
    assert bwd(lib, ptrs) == _lib.FA_ERR_ALIGNMENT


def test_bwd_bad_shape(lib):
    assert bwd(lib, B=0) == _lib.FA_ERR_INVALID_ARG
    assert bwd(lib, d=96, ws_bytes=1 << 30) == _lib.FA_ERR_UNSUPPORTED
    assert bwd(lib, scale=float("nan")) == _lib.FA_ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(lib) == _lib.FA_ERR_CUDA
    assert _lib.last_cuda_error() != 0
    assert lib.fa_get_device_status(None) == _lib.FA_ERR_CUDA


def test_python_binding_raises_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()


@pytest.mark.parametrize("H,Hkv", [(8, 3), (4, 0), (4, -1), (2, 4)])
def test_gqa_head_counts_checked(lib, H, Hkv):
    st = lib.fa_fwd_gqa(A, A, A, A, A, 1, H, Hkv, 128, 128, ctypes.c_float(0.1), 1, None)
    assert st == _lib.FA_ERR_INVALID_ARG
    ws = lib.fa_bwd_workspace_size(1, H, 128, 128) or (1 << 20)
    st = lib.fa_bwd_gqa(*([A] * 9), W, ws, 1, H, Hkv, 128, 128, ctypes.c_float(0.1), 1, None)
    assert st == _lib.FA_ERR_INVALID_ARG


def test_gqa_valid_heads_pass_host_checks(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fa_fwd_gqa(A, A, A, A, A, 1, 8, 2, 128, 128, ctypes.c_float(0.1), 1, None) == _lib.FA_ERR_CUDA


def bwd_det(lib, ptrs=None, ws=W, ws_bytes=None, B=1, H=2, Hkv=1, N=128, d=128, scale=0.1):
    p = [A] * 9 if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = lib.fa_bwd_deterministic_workspace_size(B, H, N, d) if B > 0 and H > 0 and N > 0 else 0
    return lib.fa_bwd_deterministic(*p, ws, ws_bytes, B, H, Hkv, N, d, ctypes.c_float(scale), 1, None)


def test_deterministic_workspace_size(lib):
    B, H, N, d = 2, 3, 300, 64
    vec = -(-(B * H * 384 * 4) // 256) * 256
    assert lib.fa_bwd_deterministic_workspace_size(B, H, N, d) == 2 * vec
    assert lib.fa_bwd_deterministic_workspace_size(B, H, N, d) < lib.fa_bwd_workspace_size(B, H, N, d)
    assert lib.fa_bwd_deterministic_workspace_size(0, 1, 8, 64) == 0
    assert lib.fa_bwd_deterministic_workspace_size(1, 1, 8, 96) == 0


@pytest.mark.parametrize("which", range(9))
def test_deterministic_null_pointer(lib, which):
    ptrs = [A] * 9
    ptrs[which] = None
    assert bwd_det(lib, ptrs) == _lib.FA_ERR_INVALID_ARG


def test_deterministic_host_checks(lib):
    assert bwd_det(lib, ws=None) == _lib.FA_ERR_WORKSPACE
    need = lib.fa_bwd_deterministic_workspace_size(1, 2, 128, 128)
    assert bwd_det(lib, ws_bytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert bwd_det(lib, ws=W + 16) == _lib.FA_ERR_ALIGNMENT
    assert bwd_det(lib, ptrs=[A] * 8 + [A + 8]) == _lib.FA_ERR_ALIGNMENT
    assert bwd_det(lib, Hkv=3) == _lib.FA_ERR_INVALID_ARG
    assert bwd_det(lib, d=96, ws_bytes=1 << 30) == _lib.FA_ERR_UNSUPPORTED
    assert bwd_det(lib, scale=float("inf")) == _lib.FA_ERR_INVALID_ARG


def test_deterministic_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert bwd_det(lib) == _lib.FA_ERR_CUDA


def dec(lib, ptrs=None, ws=W, ws_bytes=None, B=1, H=4, Hkv=2, Nk=1000, d=128, scale=0.1, chunks=0):
    p = [A] * 5 if ptrs is None else ptrs
    if ws_bytes is None:
        ws_bytes = lib.fa_decode_workspace_size(B, H, Hkv, Nk, d) or (1 << 20)
    return lib.fa_decode(*p, ws, ws_bytes, B, H, Hkv, Nk, d, ctypes.c_float(scale), chunks, None)


def test_decode_workspace_size(lib):
    B, H, Nk, d = 2, 8, 1000, 128           # 16 stages of 64 keys -> 16 chunk slots
    slots = B * H * 16
    vec = -(-(slots * 4) // 256) * 256
    assert lib.fa_decode_workspace_size(B, H, 2, Nk, d) == 2 * vec + slots * d * 4
    big = lib.fa_decode_workspace_size(1, 1, 1, 1 << 20, 64)   # capped at 256 chunks
    assert big == 2 * 1024 + 256 * 64 * 4
    assert lib.fa_decode_workspace_size(1, 4, 3, 100, 128) == 0      # Hkv does not divide H
    assert lib.fa_decode_workspace_size(1, 34, 2, 100, 128) == 0     # group of 17
    assert lib.fa_decode_workspace_size(1, 32, 2, 100, 128) > 0      # group of 16
    assert lib.fa_decode_workspace_size(1, 4, 2, 100, 96) == 0


@pytest.mark.parametrize("which", range(5))
def test_decode_null_pointer(lib, which):
    ptrs = [A] * 5
    ptrs[which] = None
    assert dec(lib, ptrs) == _lib.FA_ERR_INVALID_ARG


def test_decode_host_checks(lib):
    assert dec(lib, ws=None) == _lib.FA_ERR_WORKSPACE
    need = lib.fa_decode_workspace_size(1, 4, 2, 1000, 128)
    assert dec(lib, ws_bytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert dec(lib, ws=W + 64) == _lib.FA_ERR_ALIGNMENT
    assert dec(lib, ptrs=[A, A, A + 8, A, A]) == _lib.FA_ERR_ALIGNMENT
    assert dec(lib, Hkv=3) == _lib.FA_ERR_INVALID_ARG
    assert dec(lib, H=34, Hkv=2) == _lib.FA_ERR_UNSUPPORTED
    assert dec(lib, d=96) == _lib.FA_ERR_UNSUPPORTED
    assert dec(lib, Nk=0) == _lib.FA_ERR_INVALID_ARG
    assert dec(lib, scale=float("nan")) == _lib.FA_ERR_INVALID_ARG
    assert dec(lib, chunks=-1) == _lib.FA_ERR_INVALID_ARG


def test_decode_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert dec(lib) == _lib.FA_ERR_CUDA


def test_fp8_host_checks(lib):
    assert lib.fa_fp8_v_bytes(2, 3, 100, 128) == 2 * 3 * 128 * 112
    assert lib.fa_fp8_v_bytes(1, 1, 16, 96) == 0
    s = ctypes.c_float(0.1)
    # null pointers
    assert lib.fa_quantize_qk_fp8(None, None, A, A, 1, 1, 128, 128, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_v_fp8(A, None, A, 1, 1, 128, 128, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_fp8(A, A, A, A, A, None, A, A, 1, 1, 1, 128, 128, s, 1, None) == _lib.FA_ERR_INVALID_ARG
    # shapes, head dims, alignment
    assert lib.fa_quantize_qk_fp8(A, None, A, A, 1, 1, 128, 96, None) == _lib.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_fp8(A, A, A, A, A, A, A, A, 1, 1, 1, 128, 64, s, 1, None) == _lib.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_fp8(A, A, A, A, A, A, A, A, 1, 4, 3, 128, 128, s, 1, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_fp8(A + 8, A, A, A, A, A, A, A, 1, 1, 1, 128, 128, s, 1, None) == _lib.FA_ERR_ALIGNMENT
    assert lib.fa_quantize_qk_fp8(A, A + 2, A, A, 1, 1, 128, 128, None) == _lib.FA_ERR_ALIGNMENT
    assert lib.fa_fwd_fp8(A, A, A, A, A, A, A, A, 1, 1, 1, 128, 128, ctypes.c_float(float("nan")), 1,
                          None) == _lib.FA_ERR_INVALID_ARG


def test_fp8_valid_calls_without_gpu_report_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.fa_quantize_qk_fp8(A, None, A, A, 1, 1, 128, 128, None) == _lib.FA_ERR_CUDA
    assert lib.fa_fwd_fp8(A, A, A, A, A, A, A, A, 1, 1, 1, 128, 128, ctypes.c_float(0.1), 1, None) == _lib.FA_ERR_CUDA


def host_step(lib, ptrs=None, buf=W, buf_bytes=None, B=1, H=2, N=128, d=128, scale=0.1, chunk=1):
    ptrs = [A] * 9 if ptrs is None else ptrs
    if buf_bytes is None:
        buf_bytes = lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, chunk)
    return lib.fa_fwd_bwd_host(*ptrs, buf, buf_bytes, B, H, N, d, ctypes.c_float(scale), 1, chunk, None)


def test_fwd_bwd_host_buffer_size(lib):
    B, H, N, d = 2, 3, 300, 64
    tensor = -(-(2 * N * d * 2) // 256) * 256           # a chunk of two heads, bf16
    lse = -(-(2 * N * 4) // 256) * 256
    ws = -(-lib.fa_bwd_workspace_size(1, 2, N, d) // 256) * 256
    assert lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, 2) == 3 * (8 * tensor + lse + ws)
    # chunk_heads <= 0 takes ceil(B*H / 8) = 1 head; above B*H it is clamped
    assert lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, 0) == lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, 1)
    assert lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, 99) == lib.fa_fwd_bwd_host_buffer_size(B, H, N, d, 6)
    assert lib.fa_fwd_bwd_host_buffer_size(0, 1, 8, 64, 1) == 0
    assert lib.fa_fwd_bwd_host_buffer_size(1, 1, 8, 96, 1) == 0


@pytest.mark.parametrize("which", range(9))
def test_fwd_bwd_host_null_pointer(lib, which):
    ptrs = [A] * 9
    ptrs[which] = None
    assert host_step(lib, ptrs) == _lib.FA_ERR_INVALID_ARG


def test_fwd_bwd_host_checks(lib):
    assert host_step(lib, B=0, buf_bytes=1 << 30) == _lib.FA_ERR_INVALID_ARG
    assert host_step(lib, d=96, buf_bytes=1 << 30) == _lib.FA_ERR_UNSUPPORTED
    assert host_step(lib, scale=float("inf")) == _lib.FA_ERR_INVALID_ARG
    assert host_step(lib, buf=None) == _lib.FA_ERR_WORKSPACE
    need = lib.fa_fwd_bwd_host_buffer_size(1, 2, 128, 128, 1)
    assert host_step(lib, buf_bytes=need - 1) == _lib.FA_ERR_WORKSPACE
    assert host_step(lib, buf=W + 16) == _lib.FA_ERR_ALIGNMENT
    # host pointers need no particular alignment
    ptrs = [A + 1] * 9
    import torch
    if not torch.cuda.is_available():
        assert host_step(lib, ptrs) == _lib.FA_ERR_CUDA


def test_fwd_bwd_host_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert host_step(lib) == _lib.FA_ERR_CUDA
    assert _lib.last_cuda_error() != 0


def _largest_n_within(lib, limit, B, H, d):
    """The largest N whose fa_bwd workspace fits in `limit` bytes (binary search)."""
    lo, hi = 1, 1 << 24
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if lib.fa_bwd_workspace_size(B, H, mid, d) <= limit:
            lo = mid
        else:
            hi = mid - 1
    return lo


@pytest.mark.parametrize("B,H,d", [(1, 4, 128), (2, 3, 64)])
def test_noalloc_limit_is_exact(lib, B, H, d):
    """fa_bwd_noalloc takes every problem whose workspace fits its built-in array and
    rejects, on the host before any launch, the next size up."""
    limit = _lib.NOALLOC_SCRATCH_BYTES
    n = _largest_n_within(lib, limit, B, H, d)
    assert lib.fa_bwd_workspace_size(B, H, n, d) <= limit < lib.fa_bwd_workspace_size(B, H, n + 1, d)
    st = lib.fa_bwd_noalloc(*([A] * 9), B, H, n + 1, d, ctypes.c_float(0.1), 1, None)
    assert st == _lib.FA_ERR_WORKSPACE
