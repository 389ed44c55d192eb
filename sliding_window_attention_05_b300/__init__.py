"""Python binding of libswa.so: SWA(w, s) prefill, ring-cache append and decode
on NVIDIA B300 (sm_103a).

The functions below only marshal arguments (shape checks, pointers, the
current CUDA stream) and call the C ABI declared in ``include/swa.h``; every
step of the computation runs in the library's CUDA kernels. There is no CPU
or PyTorch fallback: if ``libswa.so`` is missing, importing this package
raises ImportError (build it with ``python sliding_window_attention_05_b300/build.py``).

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswa.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "swa.h")

SWA_OK = 0
SWA_ERR_INVALID_ARG = 1
SWA_ERR_UNSUPPORTED = 2
SWA_ERR_CUDA = 3
SWA_ERR_DEVICE = 4

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python sliding_window_attention_05_b300/build.py`"
        " (the SWA kernels have no fallback)")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_lib.swa_prefill.restype = _i
_lib.swa_prefill.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp]
_lib.swa_prefill_lse.restype = _i
_lib.swa_prefill_lse.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp]
_lib.swa_prefill_backward_workspace_size.restype = _sz
_lib.swa_prefill_backward_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.swa_prefill_backward.restype = _i
_lib.swa_prefill_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                      _i, _i, _i, _f, _vp, _sz, _vp]
_lib.swa_cache_append.restype = _i
_lib.swa_cache_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp]
_lib.swa_decode_workspace_size.restype = _sz
_lib.swa_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
_lib.swa_decode.restype = _i
_lib.swa_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]
_lib.swa_append_decode.restype = _i
_lib.swa_append_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f,
                                   _vp, _sz, _vp]
_lib.swa_prefill_chunk_workspace_size.restype = _sz
_lib.swa_prefill_chunk_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i, _i, ctypes.c_longlong]
_lib.swa_prefill_chunk.restype = _i
_lib.swa_prefill_chunk.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                   ctypes.c_longlong, _f, _vp, _sz, _vp]
_lib.swa_page_pool_create.restype = _vp
_lib.swa_page_pool_create.argtypes = [_i]
_lib.swa_page_pool_destroy.restype = None
_lib.swa_page_pool_destroy.argtypes = [_vp]
_lib.swa_page_pool_free_pages.restype = _i
_lib.swa_page_pool_free_pages.argtypes = [_vp]
_lib.swa_paged_reserve.restype = _i
_lib.swa_paged_reserve.argtypes = [_vp, _vp, _i, ctypes.c_longlong, _i, _i, _i]
_lib.swa_paged_reserve_range.restype = _i
_lib.swa_paged_reserve_range.argtypes = [_vp, _vp, _i, ctypes.c_longlong, ctypes.c_longlong, _i,
                                         _i, _i]
_lib.swa_paged_prefill_chunk.restype = _i
_lib.swa_paged_prefill_chunk.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                         _i, _i, _i, _i, ctypes.c_longlong, _f, _vp, _sz, _vp]
_lib.swa_paged_release.restype = _i
_lib.swa_paged_release.argtypes = [_vp, _vp, _i]
_lib.swa_paged_append.restype = _i
_lib.swa_paged_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                                  _i, _vp]
_lib.swa_paged_decode.restype = _i
_lib.swa_paged_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                  _f, _vp, _sz, _vp]
_lib.swa_decode_noalloc.restype = _i
_lib.swa_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]
_lib.swa_debug_decode_timeout.restype = _i
_lib.swa_debug_decode_timeout.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp,
                                          _sz, ctypes.c_ulonglong, _i, _vp]
_lib.swa_cache_slot.restype = ctypes.c_longlong
_lib.swa_cache_slot.argtypes = [ctypes.c_longlong, _i, _i]
_lib.swa_cache_bytes.restype = _sz
_lib.swa_cache_bytes.argtypes = [_i, _i, _i, _i, _i]
_lib.swa_prefill_plan.restype = _i
_lib.swa_prefill_plan.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.POINTER(_i)]
_lib.swa_prefill_select.restype = _i
_lib.swa_prefill_select.argtypes = [_i]
_lib.swa_debug_keymask.restype = _i
_lib.swa_debug_keymask.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp]
_lib.swa_keymask_host.restype = _i
_lib.swa_keymask_host.argtypes = [_i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp]
_lib.swa_device_error.restype = _i
_lib.swa_device_error.argtypes = [ctypes.POINTER(_i), _i]
_lib.swa_status_string.restype = ctypes.c_char_p
_lib.swa_status_string.argtypes = [_i]
_lib.swa_last_error.restype = ctypes.c_char_p
_lib.swa_last_error.argtypes = []


class SwaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.swa_last_error().decode(errors="replace")
        super().__init__(f"{where}: {_lib.swa_status_string(status).decode()} ({msg})")


def _check(status: int, where: str):
    if status != SWA_OK:
        raise SwaError(status, where)


def lib() -> ctypes.CDLL:
    """The loaded libswa.so (for calling the C ABI directly)."""
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/swa.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z0-9_]+)\s*\(", text)))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _bf16_cuda(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _expect_shape(t: torch.Tensor | None, shape, name: str):
    """Raise ValueError unless t (if given) has exactly this shape."""
    if t is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ndim(t: torch.Tensor, n: int, name: str):
    if t.dim() != n:
        raise ValueError(f"{name} must have {n} dimensions, got shape {tuple(t.shape)}")


def _check_cache(kcache: torch.Tensor, vcache: torch.Tensor, B: int, d: int, w: int, s: int):
    """The ring cache of these sizes: K and V [B, Hkv, s + w, d] (the library
    derives its strides from w and s alone, so any other shape would be read or
    written out of bounds)."""
    _ndim(kcache, 4, "kcache")
    want = (B, kcache.shape[1], int(s) + int(w), d)
    _expect_shape(kcache, want, "kcache ([B, Hkv, s + w, d])")
    _expect_shape(vcache, want, "vcache ([B, Hkv, s + w, d])")


def _check_pos(pos: torch.Tensor, B: int, name: str = "pos"):
    _expect_shape(pos, (B,), name)
    if pos.dtype != torch.int32 or not pos.is_cuda:
        raise TypeError(f"{name} must be a CUDA int32 tensor")


def _default_scale(d: int, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


# ---------------------------------------------------------------- prefill

def swa_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, w: int, s: int,
                scale: float | None = None, out: torch.Tensor | None = None, stream=None,
                lse: torch.Tensor | None = None):
    """SWA(w, s) prefill. q [B,L,Hq,d], k/v [B,L,Hkv,d] bf16 -> out [B,L,Hq,d].

    CUDA tensors run asynchronously on the current stream. CPU tensors are the
    host-buffer path: they are copied to the current device, the kernel runs,
    and the result is copied back to a (pinned) host tensor before returning.
    lse (CUDA fp32 [B, Hq, L], optional) also receives each row's log-sum-exp
    (swa_prefill_lse), which swa_prefill_backward needs.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _ndim(t, 4, n)
    B, L, Hq, d = q.shape
    if k.shape[:2] != (B, L) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    _expect_shape(out, q.shape, "out")
    if lse is not None:
        _expect_shape(lse, (B, Hq, L), "lse")
        if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
            raise TypeError("lse must be a contiguous CUDA float32 tensor")
    if not q.is_cuda:
        if lse is not None:
            raise ValueError("lse is supported with CUDA tensors only")
        dev = torch.device("cuda", torch.cuda.current_device())
        qd, kd, vd = (x.to(dev, non_blocking=True) for x in (q, k, v))
        od = swa_prefill(qd, kd, vd, w, s, scale, None, stream)
        host = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        host.copy_(od, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return host
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _bf16_cuda(t, n)
    Hkv = k.shape[2]
    if out is None:
        out = torch.empty_like(q)
    else:
        _bf16_cuda(out, "out")
    if lse is not None:
        _check(_lib.swa_prefill_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, L, Hq,
                                    Hkv, d, int(w), int(s), _default_scale(d, scale),
                                    _stream(stream)), "swa_prefill_lse")
        return out
    _check(_lib.swa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, L, Hq, Hkv, d, int(w),
                            int(s), _default_scale(d, scale), _stream(stream)), "swa_prefill")
    return out


def swa_prefill_backward_workspace_size(B: int, L: int, Hq: int, Hkv: int, d: int, s: int) -> int:
    return int(_lib.swa_prefill_backward_workspace_size(B, L, Hq, Hkv, d, s))


def swa_prefill_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                         dout: torch.Tensor, lse: torch.Tensor, w: int, s: int,
                         scale: float | None = None, dq=None, dk=None, dv=None, workspace=None,
                         stream=None):
    """Gradients (dq [B,L,Hq,d], dk, dv [B,L,Hkv,d], bf16) of the SWA(w, s)
    prefill for the upstream gradient dout [B,L,Hq,d]; out and lse are the
    forward's output and row log-sum-exp (swa_prefill(..., lse=...))."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _ndim(t, 4, n)
    B, L, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, L, Hkv, d) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    _expect_shape(out, q.shape, "out")
    _expect_shape(dout, q.shape, "dout")
    _expect_shape(lse, (B, Hq, L), "lse")
    _expect_shape(dq, q.shape, "dq")
    _expect_shape(dk, k.shape, "dk")
    _expect_shape(dv, k.shape, "dv")
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _bf16_cuda(t, n)
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise TypeError("lse must be a contiguous CUDA float32 tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = swa_prefill_backward_workspace_size(B, L, Hq, Hkv, d, s)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(_lib.swa_prefill_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, L, Hq, Hkv, d, int(w),
                                     int(s), _default_scale(d, scale), _ptr(workspace), wbytes,
                                     _stream(stream)), "swa_prefill_backward")
    return dq, dk, dv


prefill = swa_prefill


def swa_prefill_plan(L: int, Hq: int, Hkv: int, d: int, w: int, s: int) -> dict:
    plan = (_i * 8)()
    _check(_lib.swa_prefill_plan(L, Hq, Hkv, d, w, s, plan), "swa_prefill_plan")
    keys = ("Tq", "rows", "n_band", "s_box", "n_sink", "stages", "ctas", "smem_bytes")
    return dict(zip(keys, list(plan)))


# ---------------------------------------------------------------- ring cache

def swa_cache_slot(pos: int, w: int, s: int) -> int:
    return int(_lib.swa_cache_slot(int(pos), int(w), int(s)))


def swa_cache_bytes(B: int, Hkv: int, d: int, w: int, s: int) -> int:
    return int(_lib.swa_cache_bytes(B, Hkv, d, w, s))


def swa_cache_append(k_new: torch.Tensor, v_new: torch.Tensor, kcache: torch.Tensor,
                     vcache: torch.Tensor, pos_start: torch.Tensor, w: int, s: int, stream=None):
    """Append tokens k_new/v_new [B,T,Hkv,d] at positions pos_start[b] + i."""
    _ndim(k_new, 4, "k_new")
    B, T, Hkv, d = k_new.shape
    _expect_shape(v_new, k_new.shape, "v_new")
    if kcache.shape != (B, Hkv, s + w, d) or vcache.shape != kcache.shape:
        raise ValueError(f"cache must be [B, Hkv, s + w, d] = {(B, Hkv, s + w, d)}")
    _check_pos(pos_start, B, "pos_start")
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (kcache, "kcache"), (vcache, "vcache")):
        _bf16_cuda(t, n)
    _check(_lib.swa_cache_append(_ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache),
                                 _ptr(pos_start), B, T, Hkv, d, int(w), int(s), _stream(stream)),
           "swa_cache_append")


def swa_decode_workspace_size(B: int, Hq: int, Hkv: int, d: int, w: int, s: int) -> int:
    return int(_lib.swa_decode_workspace_size(B, Hq, Hkv, d, w, s))


def swa_decode(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor, pos: torch.Tensor,
               w: int, s: int, scale: float | None = None, out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, stream=None):
    """One decode step: q [B,Hq,d] over the ring cache holding position pos[b]."""
    _ndim(q, 3, "q")
    B, Hq, d = q.shape
    _check_cache(kcache, vcache, B, d, w, s)
    _expect_shape(out, q.shape, "out")
    _check_pos(pos, B)
    for t, n in ((q, "q"), (kcache, "kcache"), (vcache, "vcache")):
        _bf16_cuda(t, n)
    Hkv = kcache.shape[1]
    if out is None:
        out = torch.empty_like(q)
    need = swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.swa_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(pos), _ptr(out), B, Hq, Hkv,
                           d, int(w), int(s), _default_scale(d, scale), _ptr(workspace), wbytes,
                           _stream(stream)), "swa_decode")
    return out


def swa_append_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      kcache: torch.Tensor, vcache: torch.Tensor, pos: torch.Tensor, w: int, s: int,
                      scale: float | None = None, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """Append the token k_new/v_new [B,Hkv,d] at position pos[b], then decode
    q [B,Hq,d] over the cache (one launch)."""
    _ndim(q, 3, "q")
    B, Hq, d = q.shape
    _check_cache(kcache, vcache, B, d, w, s)
    Hkv = kcache.shape[1]
    if k_new.shape != (B, Hkv, d) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be [B, Hkv, d] = {(B, Hkv, d)}")
    _expect_shape(out, q.shape, "out")
    _check_pos(pos, B)
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (kcache, "kcache"),
                 (vcache, "vcache")):
        _bf16_cuda(t, n)
    if out is None:
        out = torch.empty_like(q)
    need = swa_decode_workspace_size(B, Hq, Hkv, d, w, s)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.swa_append_decode(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache),
                                  _ptr(pos), _ptr(out), B, Hq, Hkv, d, int(w), int(s),
                                  _default_scale(d, scale), _ptr(workspace), wbytes,
                                  _stream(stream)), "swa_append_decode")
    return out


def swa_prefill_chunk_workspace_size(B: int, T: int, Hq: int, Hkv: int, d: int, w: int, s: int,
                                     pos0: int) -> int:
    return int(_lib.swa_prefill_chunk_workspace_size(B, T, Hq, Hkv, d, w, s, int(pos0)))


def swa_prefill_chunk(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      kcache: torch.Tensor, vcache: torch.Tensor, pos0: int, w: int, s: int,
                      scale: float | None = None, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None):
    """Prefill the chunk q [B,T,Hq,d], k_new/v_new [B,T,Hkv,d] at positions
    pos0 .. pos0+T-1 against the ring cache, then append it; returns out [B,T,Hq,d]."""
    _ndim(q, 4, "q")
    B, T, Hq, d = q.shape
    _check_cache(kcache, vcache, B, d, w, s)
    Hkv = kcache.shape[1]
    if k_new.shape != (B, T, Hkv, d) or v_new.shape != k_new.shape:
        raise ValueError(f"k_new/v_new must be [B, T, Hkv, d] = {(B, T, Hkv, d)}")
    _expect_shape(out, q.shape, "out")
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (kcache, "kcache"),
                 (vcache, "vcache")):
        _bf16_cuda(t, n)
    if out is None:
        out = torch.empty_like(q)
    need = swa_prefill_chunk_workspace_size(B, T, Hq, Hkv, d, w, s, pos0)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(_lib.swa_prefill_chunk(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(kcache), _ptr(vcache),
                                  _ptr(out), B, T, Hq, Hkv, d, int(w), int(s), int(pos0),
                                  _default_scale(d, scale), _ptr(workspace), wbytes,
                                  _stream(stream)), "swa_prefill_chunk")
    return out


cache_append = swa_cache_append
prefill_chunk = swa_prefill_chunk
decode = swa_decode
append_decode = swa_append_decode


class RingCache:
    """A rolling KV cache of s sink slots + w window slots per (sequence, KV
    head), in device memory owned by this object (allocated through PyTorch)."""

    def __init__(self, B: int, Hkv: int, d: int, w: int, s: int, device=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.B, self.Hkv, self.d, self.w, self.s = B, Hkv, d, w, s
        self.k = torch.zeros(B, Hkv, s + w, d, dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)
        # position the next appended token gets, per sequence (on the device, so
        # that a CUDA graph of steps replays with advancing positions)
        self.next_pos = torch.zeros(B, dtype=torch.int32, device=device)
        self._last_pos = torch.zeros(B, dtype=torch.int32, device=device)
        self._workspace = None
        self._chunk_ws = None
        # host copy of next_pos for the chunked prefill (which needs pos0 on the
        # host); every method below keeps both in step
        self.length = 0

    def _workspace_for(self, q: torch.Tensor):
        B, Hq, d = q.shape
        need = swa_decode_workspace_size(B, Hq, self.Hkv, d, self.w, self.s)
        if need and (self._workspace is None or self._workspace.numel() < need):
            self._workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        return self._workspace if need else None

    def seek(self, pos: int):
        """Make pos the position the next appended token gets, for every
        sequence (e.g. to fill only the slots a later position still needs)."""
        self.next_pos.fill_(int(pos))
        self.length = int(pos)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Append [B, T, Hkv, d] tokens after the ones already held."""
        T = k_new.shape[1]
        swa_cache_append(k_new, v_new, self.k, self.v, self.next_pos, self.w, self.s, stream)
        self.next_pos.add_(T)
        self.length += T

    def prefill_chunk(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      scale: float | None = None, out=None, stream=None):
        """Attention of the next T prompt tokens (q [B,T,Hq,d], k_new/v_new
        [B,T,Hkv,d]) over the cache plus themselves; the chunk is then appended."""
        B, T, Hq, d = q.shape
        need = swa_prefill_chunk_workspace_size(B, T, Hq, self.Hkv, d, self.w, self.s, self.length)
        if self._chunk_ws is None or self._chunk_ws.numel() < need:
            self._chunk_ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        res = swa_prefill_chunk(q, k_new, v_new, self.k, self.v, self.length, self.w, self.s,
                                scale, out, self._chunk_ws, stream)
        self.next_pos.add_(T)
        self.length += T
        return res

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
             scale: float | None = None, out=None, stream=None):
        """Append one token per sequence (k_new/v_new [B, Hkv, d]) and decode
        q [B, Hq, d] at its position, in one launch."""
        ws = self._workspace_for(q)
        res = swa_append_decode(q, k_new, v_new, self.k, self.v, self.next_pos, self.w, self.s,
                                scale, out, ws, stream)
        self.next_pos.add_(1)
        self.length += 1
        return res

    def decode(self, q: torch.Tensor, scale: float | None = None, out=None, stream=None):
        """Attend q [B, Hq, d] (the newest token's queries) over the cache."""
        ws = self._workspace_for(q)
        torch.sub(self.next_pos, 1, out=self._last_pos)
        return swa_decode(q, self.k, self.v, self._last_pos, self.w, self.s, scale, out, ws, stream)


# ---------------------------------------------------------------- paged layout

class PagePool:
    """A pool of KV pages shared by layers: the host allocator (in libswa.so)
    and the device pools kpool, vpool [n_pages, Hkv, page_size, d] bf16."""

    def __init__(self, n_pages: int, Hkv: int, d: int, page_size: int = 64, device=None):
        device = device or torch.device("cuda", torch.cuda.current_device())
        handle = _lib.swa_page_pool_create(n_pages)
        if not handle:
            raise SwaError(SWA_ERR_INVALID_ARG, "swa_page_pool_create")
        self._h = ctypes.c_void_p(handle)
        self.n_pages, self.Hkv, self.d, self.page_size = n_pages, Hkv, d, page_size
        self.k = torch.zeros(n_pages, Hkv, page_size, d, dtype=torch.bfloat16, device=device)
        self.v = torch.zeros_like(self.k)

    def free_pages(self) -> int:
        return int(_lib.swa_page_pool_free_pages(self._h))

    def reserve(self, table, pos_hi: int, w: int, s: int, pos_lo: int | None = None):
        """table: host int32 tensor [max_pages] (contiguous). Maps the pages of
        K(p) for every p in [pos_lo, pos_hi] (pos_lo defaults to pos_hi)."""
        if pos_lo is None:
            _check(_lib.swa_paged_reserve(self._h, ctypes.c_void_p(table.data_ptr()),
                                          table.numel(), int(pos_hi), int(w), int(s),
                                          self.page_size), "swa_paged_reserve")
        else:
            _check(_lib.swa_paged_reserve_range(self._h, ctypes.c_void_p(table.data_ptr()),
                                                table.numel(), int(pos_lo), int(pos_hi), int(w),
                                                int(s), self.page_size),
                   "swa_paged_reserve_range")

    def release(self, table):
        _check(_lib.swa_paged_release(self._h, ctypes.c_void_p(table.data_ptr()), table.numel()),
               "swa_paged_release")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.swa_page_pool_destroy(h)
            self._h = None


class PagedKVCache:
    """One layer's KV cache in the pages of a shared PagePool: SWA(w, s)
    layers keep the pages of the sinks and the last w positions, full layers
    (w beyond every position) keep every page. Positions advance together for
    the B sequences; the page tables are kept on the host and copied to the
    device whenever they change."""

    def __init__(self, pool: PagePool, B: int, w: int, s: int, max_len: int):
        self.pool, self.B, self.w, self.s = pool, B, w, s
        self.max_pages = (max_len + pool.page_size - 1) // pool.page_size
        # pageable on purpose: a copy from it takes its contents at the call,
        # so the next step's reserve cannot change what this step's kernels see
        self.table = torch.full((B, self.max_pages), -1, dtype=torch.int32)
        device = pool.k.device
        self.table_dev = torch.full((B, self.max_pages), -1, dtype=torch.int32, device=device)
        self.length = 0
        self.pos_dev = torch.zeros(B, dtype=torch.int32, device=device)
        self._pos_value = 0          # what pos_dev holds (set only when it changes)
        self._workspace = None
        self._chunk_ws = None

    def _set_pos(self, value: int):
        if value != self._pos_value:
            self.pos_dev.fill_(value)
            self._pos_value = value

    def _reserve(self, pos_hi: int, pos_lo: int | None = None):
        for b in range(self.B):
            self.pool.reserve(self.table[b], pos_hi, self.w, self.s, pos_lo)
        self.table_dev.copy_(self.table)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None):
        """Append [B, T, Hkv, d] tokens at positions length .. length + T - 1."""
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _bf16_cuda(t, n)
        B, T, Hkv, d = k_new.shape
        self._reserve(self.length + T - 1)
        self._set_pos(self.length)
        _check(_lib.swa_paged_append(_ptr(k_new), _ptr(v_new), _ptr(self.pool.k), _ptr(self.pool.v),
                                     _ptr(self.table_dev), _ptr(self.pos_dev), B, T, Hkv, d,
                                     self.pool.page_size, self.max_pages, self.pool.n_pages,
                                     self.w, self.s, _stream(stream)), "swa_paged_append")
        self.length += T

    def prefill_chunk(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      scale: float | None = None, out=None, stream=None):
        """Attention of the next T prompt tokens (q [B,T,Hq,d], k_new/v_new
        [B,T,Hkv,d]) over the pages plus themselves; the chunk is then appended."""
        _ndim(q, 4, "q")
        B, T, Hq, d = q.shape
        Hkv = self.pool.Hkv
        _expect_shape(k_new, (self.B, T, Hkv, self.pool.d), "k_new")
        _expect_shape(v_new, (self.B, T, Hkv, self.pool.d), "v_new")
        _expect_shape(out, q.shape, "out")
        for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
            _bf16_cuda(t, n)
        if out is None:
            out = torch.empty_like(q)
        pos0 = self.length
        self._reserve(pos0 + T - 1, pos0)
        need = swa_prefill_chunk_workspace_size(B, T, Hq, Hkv, d, self.w, self.s, pos0)
        if self._chunk_ws is None or self._chunk_ws.numel() < need:
            self._chunk_ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        _check(_lib.swa_paged_prefill_chunk(
            _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(self.pool.k), _ptr(self.pool.v),
            _ptr(self.table_dev), _ptr(out), B, T, Hq, Hkv, d, self.pool.page_size,
            self.max_pages, self.pool.n_pages, self.w, self.s, pos0, _default_scale(d, scale),
            _ptr(self._chunk_ws), self._chunk_ws.numel(), _stream(stream)),
            "swa_paged_prefill_chunk")
        self.length += T
        return out

    def decode(self, q: torch.Tensor, scale: float | None = None, out=None, stream=None):
        """q [B, Hq, d]: attend at the newest position (length - 1)."""
        _bf16_cuda(q, "q")
        B, Hq, d = q.shape
        need = swa_decode_workspace_size(B, Hq, self.pool.Hkv, d, self.w, self.s)
        if need and (self._workspace is None or self._workspace.numel() < need):
            self._workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws = self._workspace if need else None
        if out is None:
            out = torch.empty_like(q)
        self._set_pos(self.length - 1)
        wbytes = 0 if ws is None else ws.numel()
        _check(_lib.swa_paged_decode(_ptr(q), _ptr(self.pool.k), _ptr(self.pool.v),
                                     _ptr(self.table_dev), _ptr(self.pos_dev), _ptr(out), B, Hq,
                                     self.pool.Hkv, d, self.pool.page_size, self.max_pages,
                                     self.pool.n_pages, self.w, self.s, _default_scale(d, scale),
                                     _ptr(ws), wbytes, _stream(stream)), "swa_paged_decode")
        return out

    def pages_held(self) -> int:
        return int((self.table >= 0).sum())

    def release(self):
        for b in range(self.B):
            self.pool.release(self.table[b])
        self.table_dev.fill_(-1)
        self.length = 0


# ---------------------------------------------------------------- test aids

PREFILL_AUTO, PREFILL_SINGLE, PREFILL_PAIR = 0, 1, 2


def swa_prefill_select(mode: int) -> int:
    """Test aid: which prefill kernel runs (PREFILL_AUTO: the library's choice,
    PREFILL_SINGLE: one query block per work item, PREFILL_PAIR: two); returns
    the previous mode."""
    prev = int(_lib.swa_prefill_select(int(mode)))
    if prev < 0:
        raise ValueError(f"prefill mode {mode} is not one of 0, 1, 2")
    return prev


def swa_debug_keymask(L: int, Hq: int, Hkv: int, d: int, w: int, s: int, row0: int, nrows: int,
                      device=None):
    """Admitted (row, key) pairs of the prefill schedule, computed on the GPU:
    returns (bits uint32 [nrows, ceil(L/32)], counts int32 [nrows]) on the device."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    words = (L + 31) // 32
    bits = torch.empty(nrows, words, dtype=torch.int32, device=device)
    counts = torch.empty(nrows, dtype=torch.int32, device=device)
    _check(_lib.swa_debug_keymask(L, Hq, Hkv, d, w, s, row0, nrows, _ptr(bits), _ptr(counts),
                                  _stream(None)), "swa_debug_keymask")
    return bits, counts


def swa_keymask_host(L: int, Hq: int, Hkv: int, d: int, w: int, s: int, row0: int, nrows: int):
    """The same admitted-pair bitmask, computed by the library's host copy of
    the schedule (no GPU needed)."""
    words = (L + 31) // 32
    bits = torch.zeros(nrows, words, dtype=torch.int32)
    counts = torch.zeros(nrows, dtype=torch.int32)
    _check(_lib.swa_keymask_host(L, Hq, Hkv, d, w, s, row0, nrows, _ptr(bits), _ptr(counts)),
           "swa_keymask_host")
    return bits, counts


def swa_device_error(clear: bool = True) -> int:
    code = _i(0)
    _check(_lib.swa_device_error(ctypes.byref(code), 1 if clear else 0), "swa_device_error")
    return code.value


def swa_status_string(status: int) -> str:
    return _lib.swa_status_string(status).decode()


def swa_last_error() -> str:
    return _lib.swa_last_error().decode(errors="replace")


# the hybrid attention stack driver (sequencing only; imports the names above)
from .stack import AttentionLayer, HybridStack, hybrid_layer_windows  # noqa: E402,F401
