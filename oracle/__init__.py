"""fp64 CPU oracle for SWA(w, s) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The CUDA library and its Python binding
never import it, and it never imports them: the two sides share only the seeded
input generators in ``swa_inputs``.

The arithmetic lives in ``swa_oracle.c`` (plain C, double precision, one query
row at a time, key sets enumerated by brute predicate). This module compiles it
with gcc, loads it with ctypes and converts arrays.

``swa_mask`` restates the boolean-mask definition of SWA(w, s) given on the
explainer page of arXiv 2608.28444 (section "核心方法 / 1. 训练免费的 SWA(w, s)"):
row t admits the window columns max(0, t-w+1) .. t and the first s columns.
It is used only to cross-check the C key-set enumeration.

Parity status of each function (what pins it, see tests/test_oracle.py):
  keyset / keymask   pinned: explicit boolean mask, closed-form counts, w>=L, s=0
  prefill            pinned: torch fp64 SDPA with the same boolean mask (library),
                     w=1 identity, q=0 mean, constant-V, GQA == repeated MHA
  weights            pinned: rows sum to one; equal torch fp64 softmax (library) of
                     the scaled scores over the same boolean mask, GQA group of 3
  decode             pinned: equals the prefill row at the same position
  ring_contents      pinned: page example (W=4, 5th token evicts the 1st), holds
                     exactly K(last), 68-slot footprint
  prefill_backward   pinned: torch fp64 autograd of SDPA with the same boolean mask
                     (library), w=1 closed form, keys' gradients sum to zero,
                     Euler identity sum_j v_j.dv_j = sum_t dout_t.out_t
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lib = None
_lock = threading.Lock()

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle C source into a shared library with gcc (OpenMP)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra_flags,
           src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None, rebuild: bool = False):
    """Load (building first if needed) the oracle library; returns the CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None or rebuild:
            stale = (not os.path.exists(_LIB_PATH)
                     or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
            if rebuild or stale:
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _bind(lib):
    lib.oracle_keyset.restype = _i64
    lib.oracle_keyset.argtypes = [_i64, _i64, _i64, _p]
    lib.oracle_keymask.restype = None
    lib.oracle_keymask.argtypes = [_i64, _i64, _i64, _p]
    lib.oracle_weights.restype = _i64
    lib.oracle_weights.argtypes = [_p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.c_double, _i64, _i64, _i64, _p]
    lib.oracle_prefill.restype = ctypes.c_int
    lib.oracle_prefill.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                   ctypes.c_double, _p, _i64, _p, _p, ctypes.c_int]
    lib.oracle_prefill_backward.restype = ctypes.c_int
    lib.oracle_prefill_backward.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64,
                                            _i64, ctypes.c_double, _p, _p, _p, ctypes.c_int]
    lib.oracle_decode.restype = ctypes.c_int
    lib.oracle_decode.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                                  ctypes.c_double, _p, _p]
    lib.oracle_ring_contents.restype = None
    lib.oracle_ring_contents.argtypes = [_i64, _i64, _i64, _p]
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(t) -> np.ndarray:
    """bf16 tensor (or uint16 array of bf16 patterns) -> contiguous uint16 array."""
    if isinstance(t, torch.Tensor):
        assert t.dtype == torch.bfloat16, t.dtype
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(t)
    assert a.dtype == np.uint16
    return a


def swa_mask(L: int, w: int, s: int) -> np.ndarray:
    """Boolean [L, L] mask of the page's definition, before the causal clamp:
    row t admits columns max(0, t-w+1)..t (window) and columns 0..s-1 (sinks)."""
    t = np.arange(L).reshape(-1, 1)
    j = np.arange(L).reshape(1, -1)
    window = (j >= np.maximum(0, t - w + 1)) & (j <= t)
    sinks = j < s
    return window | sinks


def keyset(t: int, w: int, s: int, lib=None) -> np.ndarray:
    lib = lib or load()
    keys = np.empty(t + 1, dtype=np.int64)
    n = lib.oracle_keyset(t, w, s, _ptr(keys))
    return keys[:n].copy()


def keymask(L: int, w: int, s: int, lib=None) -> np.ndarray:
    lib = lib or load()
    m = np.zeros((L, L), dtype=np.uint8)
    lib.oracle_keymask(L, w, s, _ptr(m))
    return m.astype(bool)


def prefill(q, k, v, w: int, s: int, scale: float, rows=None, nthreads: int = 0,
            lib=None):
    """out [B, nrows, Hq, d] and lse [B, nrows, Hq] in float64.

    q [B, L, Hq, d], k and v [B, L, Hkv, d] bf16; rows = query positions to
    compute (default all). The scale is rounded to float32 first, as the CUDA
    library receives it."""
    lib = lib or load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, L, Hq, d = qb.shape
    Hkv = kb.shape[2]
    if rows is None:
        rows_arr = None
        nrows = L
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.shape[0]
    out = np.zeros((B, nrows, Hq, d), dtype=np.float64)
    lse = np.zeros((B, nrows, Hq), dtype=np.float64)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_prefill(_ptr(qb), _ptr(kb), _ptr(vb), B, L, Hq, Hkv, d, w, s,
                            float(np.float32(scale)),
                            None if rows_arr is None else _ptr(rows_arr), nrows,
                            _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_prefill rejected its arguments (rc={rc})")
    return out, lse


def prefill_backward(q, k, v, dout, w: int, s: int, scale: float, nthreads: int = 0, lib=None):
    """(dq [B,L,Hq,d], dk, dv [B,L,Hkv,d]) in float64: the gradients of the
    prefill outputs with respect to q, k, v for the upstream gradient dout
    ([B,L,Hq,d], any float type; used in float64)."""
    lib = lib or load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, L, Hq, d = qb.shape
    Hkv = kb.shape[2]
    g = dout.detach().cpu().double().numpy() if isinstance(dout, torch.Tensor) else dout
    g = np.ascontiguousarray(g, dtype=np.float64)
    assert g.shape == (B, L, Hq, d), g.shape
    dq = np.zeros((B, L, Hq, d), dtype=np.float64)
    dk = np.zeros((B, L, Hkv, d), dtype=np.float64)
    dv = np.zeros((B, L, Hkv, d), dtype=np.float64)
    if nthreads <= 0:
        nthreads = os.cpu_count() or 1
    rc = lib.oracle_prefill_backward(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(g), B, L, Hq, Hkv, d, w,
                                     s, float(np.float32(scale)), _ptr(dq), _ptr(dk), _ptr(dv),
                                     int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_prefill_backward rejected its arguments (rc={rc})")
    return dq, dk, dv


def weights(q, k, w: int, s: int, scale: float, b: int, hq: int, t: int, lib=None):
    """Softmax weights of row (b, hq, t) over K(t), in increasing key order."""
    lib = lib or load()
    qb, kb = _bits(q), _bits(k)
    B, L, Hq, d = qb.shape
    Hkv = kb.shape[2]
    wts = np.zeros(t + 1, dtype=np.float64)
    n = lib.oracle_weights(_ptr(qb), _ptr(kb), L, Hq, Hkv, d, w, s,
                           float(np.float32(scale)), b, hq, t, _ptr(wts))
    return wts[:n].copy()


def decode(q, hist_pos, hist_k, hist_v, pos: int, w: int, s: int, scale: float, lib=None):
    """One decode row per query head: q [Hq, d]; history rows [nh, Hkv, d].
    Returns (out [Hq, d], lse [Hq]) in float64."""
    lib = lib or load()
    qb, kb, vb = _bits(q), _bits(hist_k), _bits(hist_v)
    Hq, d = qb.shape
    nh, Hkv, _ = kb.shape
    hp = np.ascontiguousarray(hist_pos, dtype=np.int64)
    out = np.zeros((Hq, d), dtype=np.float64)
    lse = np.zeros(Hq, dtype=np.float64)
    rc = lib.oracle_decode(_ptr(qb), _ptr(hp), _ptr(kb), _ptr(vb), nh, pos, Hq, Hkv, d,
                           w, s, float(np.float32(scale)), _ptr(out), _ptr(lse))
    if rc == -2:
        raise ValueError("history does not hold every position of K(pos) exactly once")
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its arguments (rc={rc})")
    return out, lse


def ring_contents(last: int, w: int, s: int, lib=None) -> np.ndarray:
    """Positions held by each of the s + w cache slots after appending 0..last."""
    lib = lib or load()
    slots = np.empty(s + w, dtype=np.int64)
    lib.oracle_ring_contents(last, w, s, _ptr(slots))
    return slots
