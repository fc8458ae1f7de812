"""Exact softmax attention for GB300 (sm_103a): forward and backward.

    o, lse = fwd(q, k, v, causal=True)            # q, k, v: [B, H, N, d] CUDA tensors
    dq, dk, dv = bwd(q, k, v, o, lse, do, causal=True)

The arithmetic runs in hand-written tcgen05/TMA kernels inside libfa_gb300.so,
reached through its C ABI (include/fa.h).  PyTorch provides device memory and
streams only.  ``build()`` compiles the library in-tree with nvcc.
"""
from __future__ import annotations

import math

import torch

from . import _lib
from ._lib import FaError  # noqa: F401

__all__ = ["fwd", "bwd", "fwd_bwd_host", "fwd_bwd_host_buffer_size", "decode", "quantize_qk_fp8", "quantize_v_fp8", "fwd_fp8", "bwd_workspace_size",
           "bwd_deterministic_workspace_size", "decode_workspace_size", "device_status", "build", "FaError"]


def build(force: bool = False) -> str:
    from .buildlib import build as _build
    return _build(force=force)


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_tensors(dtype, shape, *ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if t.dtype != dtype:
            raise ValueError(f"expected {dtype}, got {t.dtype}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"expected shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.device != ts[0].device:
            raise ValueError("tensors must be on one device")


def _shapes(q, k):
    """[B, H, N, d] queries and [B, Hkv, N, d] keys/values (Hkv divides H)."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, H, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("q and k/v must agree in B, N and d")
    Hkv = k.shape[1]
    if H % Hkv != 0:
        raise ValueError("the number of query heads must be a multiple of the key/value heads")
    return B, H, Hkv, N, d


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """O = softmax(scale * q k^T [causal mask]) v and the natural-log logsumexp per row.

    q: [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H (Hkv < H is grouped-query
    attention: query head h uses key/value head h // (H // Hkv)).  bf16 tensors use
    fa_fwd / fa_fwd_gqa; float32 tensors use fa_fwd_f32 (d = 64, Hkv = H).
    Returns (o, lse) with lse float32 [B, H, N].
    """
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q, k, v must be bfloat16 or float32")
    B, H, Hkv, N, d = _shapes(q, k)
    _check_tensors(dtype, q.shape, q)
    _check_tensors(dtype, k.shape, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_tensors(dtype, q.shape, q, out)
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    lib = _lib.load()
    stream = _stream_ptr(q.device)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr())
    if dtype == torch.float32:
        if Hkv != H:
            raise ValueError("grouped-query attention takes bfloat16 tensors")
        st, name = lib.fa_fwd_f32(*ptrs, B, H, N, d, scale, int(bool(causal)), stream), "fa_fwd_f32"
    elif Hkv == H:
        st, name = lib.fa_fwd(*ptrs, B, H, N, d, scale, int(bool(causal)), stream), "fa_fwd"
    else:
        st, name = lib.fa_fwd_gqa(*ptrs, B, H, Hkv, N, d, scale, int(bool(causal)), stream), "fa_fwd_gqa"
    _lib.check(st, name)
    return out, lse


def bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.load().fa_bwd_workspace_size(B, H, N, d))


def bwd_deterministic_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.load().fa_bwd_deterministic_workspace_size(B, H, N, d))


def bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
        dq=None, dk=None, dv=None, workspace=None, deterministic: bool = False):
    """Gradients (dq, dk, dv) of sum(o * do), recomputing the probabilities from lse.

    Shapes as in fwd; with grouped-query attention dk and dv are [B, Hkv, N, d] and sum
    the contributions of the query heads that share each key/value head.
    ``deterministic=True`` uses fa_bwd_deterministic: bit-identical results from run
    to run (dQ has one writer per row).
    """
    B, H, Hkv, N, d = _shapes(q, k)
    _check_tensors(torch.bfloat16, q.shape, q, o, do)
    _check_tensors(torch.bfloat16, k.shape, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensors(torch.bfloat16, q.shape, q, dq)
    _check_tensors(torch.bfloat16, k.shape, k, dk, dv)
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    need = (bwd_deterministic_workspace_size if deterministic else bwd_workspace_size)(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lib = _lib.load()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size())
    stream = _stream_ptr(q.device)
    if deterministic:
        st, name = (lib.fa_bwd_deterministic(*args, B, H, Hkv, N, d, scale, int(bool(causal)), stream),
                    "fa_bwd_deterministic")
    elif Hkv == H:
        st, name = lib.fa_bwd(*args, B, H, N, d, scale, int(bool(causal)), stream), "fa_bwd"
    else:
        st, name = lib.fa_bwd_gqa(*args, B, H, Hkv, N, d, scale, int(bool(causal)), stream), "fa_bwd_gqa"
    _lib.check(st, name)
    return dq, dk, dv


def fwd_bwd_host_buffer_size(B: int, H: int, N: int, d: int, chunk_heads: int = 0) -> int:
    return int(_lib.load().fa_fwd_bwd_host_buffer_size(B, H, N, d, chunk_heads))


def fwd_bwd_host(q, k, v, do, causal: bool = False, scale: float | None = None, o=None, lse=None,
                 dq=None, dk=None, dv=None, buffer=None, chunk_heads: int = 0, device=None):
    """Forward then backward on tensors in host memory (fa_fwd_bwd_host): the library
    copies chunks of heads in, runs fa_fwd and fa_bwd on them and copies the results
    out, overlapping the copies with the kernels.

    q, k, v, do: [B, H, N, d] bf16 CPU tensors (page-locked for overlap).  Returns
    (o, lse, dq, dk, dv) as CPU tensors; they are complete once the current stream of
    ``device`` has been synchronised.  ``buffer`` is the device scratch of
    fwd_bwd_host_buffer_size(B, H, N, d, chunk_heads) bytes (allocated if None).
    """
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, H, N, d = q.shape
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)

    def host(t, dtype, shape, name):
        if t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dtype} CPU tensor of shape {tuple(shape)}")
        return t

    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        host(t, torch.bfloat16, q.shape, name)
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin) if lse is None else lse
    dq = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dq is None else dq
    dk = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dk is None else dk
    dv = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dv is None else dv
    for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        host(t, torch.bfloat16, q.shape, name)
    host(lse, torch.float32, (B, H, N), "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = fwd_bwd_host_buffer_size(B, H, N, d, chunk_heads)
    if buffer is None:
        buffer = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    if not buffer.is_cuda:
        raise ValueError("buffer must be a CUDA tensor")
    lib = _lib.load()
    st = lib.fa_fwd_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), buffer.data_ptr(),
                             buffer.numel() * buffer.element_size(), B, H, N, d, scale, int(bool(causal)),
                             int(chunk_heads), _stream_ptr(buffer.device))
    _lib.check(st, "fa_fwd_bwd_host")
    return o, lse, dq, dk, dv


def decode_workspace_size(B: int, H: int, Hkv: int, Nk: int, d: int) -> int:
    return int(_lib.load().fa_decode_workspace_size(B, H, Hkv, Nk, d))


def decode(q, k, v, scale: float | None = None, out=None, lse=None, workspace=None, num_chunks: int = 0):
    """One query row per head against all keys: q [B, H, d], k and v [B, Hkv, Nk, d]
    (bf16, Hkv dividing H, H / Hkv <= 16).  Returns (o [B, H, d] bf16, lse [B, H] fp32).
    The keys are split into chunks merged on the device (num_chunks = 0: automatic)."""
    if q.dim() != 3 or k.dim() != 4:
        raise ValueError("expected q [B, H, d] and k, v [B, Hkv, Nk, d]")
    B, H, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or H % Hkv != 0:
        raise ValueError("q and k/v must agree in B and d, and Hkv must divide H")
    _check_tensors(torch.bfloat16, q.shape, q)
    _check_tensors(torch.bfloat16, k.shape, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensors(torch.bfloat16, q.shape, q, out)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H] tensor")
    if workspace is None:
        workspace = torch.empty(decode_workspace_size(B, H, Hkv, Nk, d), dtype=torch.uint8, device=q.device)
    st = _lib.load().fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                               B, H, Hkv, Nk, d, scale, int(num_chunks), _stream_ptr(q.device))
    _lib.check(st, "fa_decode")
    return out, lse


def quantize_qk_fp8(x, signs=None):
    """e4m3 codes of Q or K [B, H, N, d] (bf16) with one scale per (batch, head).  With
    ``signs`` (a float32 tensor of +-1 of length d, the same for Q and K) every row is
    first rotated by diag(signs) H / sqrt(d) (incoherent processing).  Returns
    (codes as a uint8 tensor [B, H, N, d], descale float32 [B, H])."""
    if x.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    B, H, N, d = x.shape
    _check_tensors(torch.bfloat16, x.shape, x)
    if signs is not None:
        if signs.dtype != torch.float32 or tuple(signs.shape) != (d,) or not signs.is_cuda:
            raise ValueError("signs must be a float32 CUDA tensor of length d")
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    descale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    st = _lib.load().fa_quantize_qk_fp8(x.data_ptr(), signs.data_ptr() if signs is not None else None,
                                        x8.data_ptr(), descale.data_ptr(), B, H, N, d, _stream_ptr(x.device))
    _lib.check(st, "fa_quantize_qk_fp8")
    return x8, descale


def quantize_v_fp8(v):
    """e4m3 codes of V [B, H, N, d] (bf16), transposed to [B, H, d, Npad] (keys contiguous,
    N padded to a multiple of 16 with zero codes), and descale float32 [B, H]."""
    if v.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    B, H, N, d = v.shape
    _check_tensors(torch.bfloat16, v.shape, v)
    npad = (N + 15) // 16 * 16
    vt8 = torch.empty((B, H, d, npad), dtype=torch.uint8, device=v.device)
    descale = torch.empty((B, H), dtype=torch.float32, device=v.device)
    st = _lib.load().fa_quantize_v_fp8(v.data_ptr(), vt8.data_ptr(), descale.data_ptr(), B, H, N, d,
                                       _stream_ptr(v.device))
    _lib.check(st, "fa_quantize_v_fp8")
    return vt8, descale


def fwd_fp8(q8, k8, vt8, descale_q, descale_k, descale_v, causal: bool = False, scale: float | None = None,
            out=None, lse=None):
    """Forward pass on e4m3 codes (from quantize_qk_fp8 / quantize_v_fp8; d = 128):
    returns (o bf16 [B, H, N, d], lse float32 [B, H, N])."""
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    if q8.dtype != torch.uint8 or k8.dtype != torch.uint8 or vt8.dtype != torch.uint8:
        raise ValueError("q8, k8 and vt8 must be uint8 code tensors")
    if tuple(k8.shape) != (B, Hkv, N, d) or tuple(vt8.shape) != (B, Hkv, d, (N + 15) // 16 * 16):
        raise ValueError("k8 must be [B, Hkv, N, d] and vt8 [B, Hkv, d, Npad]")
    for t in (q8, k8, vt8, descale_q, descale_k, descale_v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    st = _lib.load().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), descale_q.data_ptr(),
                                descale_k.data_ptr(), descale_v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, H, Hkv, N, d, scale, int(bool(causal)), _stream_ptr(q8.device))
    _lib.check(st, "fa_fwd_fp8")
    return out, lse


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    s = torch.cuda.current_stream() if stream is None else stream
    return int(_lib.load().fa_get_device_status(s.cuda_stream))
