"""The oracle for split-KV decode attention (Flash-Decoding).

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``split_kv_gb300``) never imports it and shares no code with
it: the oracle is the slow, plain fp64 CPU statement of the method that the
CUDA path is checked against.

Contents
--------
* ``liboracle.so`` (built from ``fd_oracle.cpp`` with g++, no CUDA): exact
  fp16/bf16 -> double conversion, plain attention (``attend``), segment states
  and their merge (``segment_state``, ``merge``, ``finalize``), the split-count
  heuristic (``plan``) and batched decode over contiguous or paged caches
  (``decode``).
* ``plan_ref.py``: a second, pure-Python statement of the split-count
  heuristic, used to cross-check both the C statement here and the library.

Citations name the pages by title and section:
  "Flash-Decoding: Split-KV Attention for Long-Context Decode" (kanthi.in) [FD];
  "Decode 专项 Attention：把长KV拆开算，再正确合并" (xuujii.github.io) [DKV].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .plan_ref import num_splits_ref, efficiency_ref  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fd_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (g++, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        d, i32, i64 = ctypes.c_double, ctypes.c_int32, ctypes.c_int64
        vp = ctypes.c_void_p
        lib.fdo_half_to_double.restype = d
        lib.fdo_half_to_double.argtypes = [ctypes.c_uint16]
        lib.fdo_bf16_to_double.restype = d
        lib.fdo_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.fdo_e4m3_to_double.restype = d
        lib.fdo_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.fdo_attend.restype = ctypes.c_int
        lib.fdo_attend.argtypes = [i64, ctypes.c_int, vp, vp, vp, d, vp, vp]
        lib.fdo_segment_state.restype = ctypes.c_int
        lib.fdo_segment_state.argtypes = [i64, ctypes.c_int, vp, vp, vp, d, vp, vp, vp]
        lib.fdo_merge.restype = ctypes.c_int
        lib.fdo_merge.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp]
        lib.fdo_finalize.restype = ctypes.c_int
        lib.fdo_finalize.argtypes = [ctypes.c_int, d, d, vp, vp, vp]
        lib.fdo_plan.restype = ctypes.c_int
        lib.fdo_plan.argtypes = [i64, i64, i64, ctypes.c_int, vp]
        lib.fdo_decode.restype = ctypes.c_int
        lib.fdo_decode.argtypes = [i32, i32, i32, i32, i32, i32, d, d, i32,
                                   vp, i64, i64, i64,
                                   vp, i64, i64, i64,
                                   vp, i64, i64, i64,
                                   vp,
                                   i32, vp, i32,
                                   vp, i64,
                                   vp, vp, i32]
        lib.fdo_hardware_threads.restype = ctypes.c_int
        lib.fdo_hardware_threads.argtypes = []
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(_load().fdo_hardware_threads())


def half_to_double(bits: int) -> float:
    return float(_load().fdo_half_to_double(int(bits) & 0xFFFF))


def bf16_to_double(bits: int) -> float:
    return float(_load().fdo_bf16_to_double(int(bits) & 0xFFFF))


def e4m3_to_double(bits: int) -> float:
    return float(_load().fdo_e4m3_to_double(int(bits) & 0xFF))


def attend(q, K, V, scale: float):
    """Plain attention of one query: returns (o[D], lse).  [FD] §1-§2."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    D = q.shape[0]
    L = K.shape[0] if K.ndim == 2 else 0
    out = np.empty(D)
    lse = np.empty(1)
    rc = _load().fdo_attend(L, D, _ptr(q), _ptr(K) if L else None, _ptr(V) if L else None,
                            float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("fdo_attend rejected its arguments")
    return out, float(lse[0])


def segment_state(q, K, V, scale: float):
    """(m, ell, u) of one key segment.  [DKV] §04."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    D = q.shape[0]
    L = K.shape[0] if K.ndim == 2 else 0
    m, ell, u = np.empty(1), np.empty(1), np.empty(D)
    rc = _load().fdo_segment_state(L, D, _ptr(q), _ptr(K) if L else None,
                                   _ptr(V) if L else None, float(scale),
                                   _ptr(m), _ptr(ell), _ptr(u))
    if rc != 0:
        raise ValueError("fdo_segment_state rejected its arguments")
    return float(m[0]), float(ell[0]), u


def merge(m, ell, u):
    """Exact merge of n states (m[n], ell[n], u[n, D]) -> (m, ell, u[D]).  [DKV] §04."""
    m, ell, u = _f64(m).reshape(-1), _f64(ell).reshape(-1), _f64(u)
    n = m.shape[0]
    D = u.shape[-1]
    mo, lo, uo = np.empty(1), np.empty(1), np.empty(D)
    rc = _load().fdo_merge(n, D, _ptr(m), _ptr(ell), _ptr(u.reshape(n, D)),
                           _ptr(mo), _ptr(lo), _ptr(uo))
    if rc != 0:
        raise ValueError("fdo_merge rejected its arguments")
    return float(mo[0]), float(lo[0]), uo


def finalize(m: float, ell: float, u):
    """(o, lse) of a state: o = u / ell, lse = m + log ell."""
    u = _f64(u)
    D = u.shape[0]
    out, lse = np.empty(D), np.empty(1)
    rc = _load().fdo_finalize(D, float(m), float(ell), _ptr(u), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("fdo_finalize rejected its arguments")
    return out, float(lse[0])


def plan(work_items: int, slots: int, n_kv_blocks: int, max_splits: int = 128,
         return_eff: bool = False):
    """Split-count heuristic of [FD] §6, C statement."""
    eff = np.empty(max_splits + 1)
    s = _load().fdo_plan(int(work_items), int(slots), int(n_kv_blocks), int(max_splits),
                         _ptr(eff))
    if s < 0:
        raise ValueError("fdo_plan rejected its arguments")
    return (int(s), eff) if return_eff else int(s)


def _bits(a) -> np.ndarray:
    """Raw 16-bit patterns of an fp16 / bf16 array (numpy uint16/float16 or torch)."""
    if hasattr(a, "detach"):  # torch tensor on the host
        import torch
        t = a.detach().contiguous()
        if t.is_cuda:
            raise ValueError("oracle inputs must be host arrays")
        return t.view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError(f"need 16-bit raw patterns, got {a.dtype}")


def _bytes8(a) -> np.ndarray:
    """Raw 8-bit patterns of an fp8 e4m3 cache (numpy uint8 or torch float8/uint8)."""
    if hasattr(a, "detach"):
        import torch
        t = a.detach().contiguous()
        if t.is_cuda:
            raise ValueError("oracle inputs must be host arrays")
        return t.view(torch.uint8).numpy()
    a = np.asarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"need 8-bit raw patterns, got {a.dtype}")
    return a


def decode(q, k, v, seqlens, *, dtype: str, n_kv_heads: int,
           page_size: int = 0, block_table=None, rows=None, n_threads: int = 0,
           kv_dtype: str | None = None, k_scale: float = 1.0, v_scale: float = 1.0):
    """Decode attention in fp64 for every (sequence, query position, query head) row.

    q: [B, Hq, D] (one query per sequence) or [B, q_len, Hq, D] (a short query
    block: position i sees the first L_b - q_len + 1 + i keys) 16-bit;
    contiguous k, v: [B, Hkv, T, D] (any 4-D strided
    view whose last dim is contiguous); paged k, v: pool [P, Hkv, page, D] (or
    any 4-D view [P, Hkv, page, D] with contiguous last dim) with block_table
    [B, max_pages] int32.  dtype: 'f16' or 'bf16', the type of q and (by
    default) of the cache.  kv_dtype='e4m3': k, v are fp8 E4M3 bytes and key /
    value j is k_scale / v_scale times the stored value (one scale per tensor).
    rows: optional flat row indices (b*q_len + i)*Hq + h.  Returns
    (out[n, D] float64, lse[n] float64).
    """
    dt = {"f16": 0, "bf16": 1}[dtype]
    kvdt = -1 if kv_dtype is None else {"f16": 0, "bf16": 1, "e4m3": 2}[kv_dtype]
    qb = _bits(q)
    if kvdt == 2:
        kb, vb = _bytes8(k), _bytes8(v)
        esz = 1
    else:
        kb, vb = _bits(k), _bits(v)
        esz = 2
    if qb.ndim == 3:
        qb = qb[:, None]
    B, q_len, Hq, D = qb.shape
    if qb.strides[-1] != 2 or kb.strides[-1] != esz or vb.strides[-1] != esz:
        raise ValueError("last dim must be contiguous")
    qs = [s // 2 for s in qb.strides]        # b, i, h, d
    ks = [s // esz for s in kb.strides]
    vs = [s // esz for s in vb.strides]
    sl = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    if sl.shape[0] != B:
        raise ValueError("seqlens must have one entry per sequence")
    bt = None
    mp = 0
    if page_size:
        bt = np.ascontiguousarray(np.asarray(block_table, dtype=np.int32))
        mp = bt.shape[1]
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows.shape[0]
    else:
        n = B * q_len * Hq
    out = np.empty((n, D))
    lse = np.empty(n)
    rc = _load().fdo_decode(
        B, Hq, int(n_kv_heads), D, dt, kvdt, float(k_scale), float(v_scale), q_len,
        qb.ctypes.data, qs[0], qs[1], qs[2],
        kb.ctypes.data, ks[0], ks[1], ks[2],
        vb.ctypes.data, vs[0], vs[1], vs[2],
        _ptr(sl),
        int(page_size), _ptr(bt) if bt is not None else None, mp,
        _ptr(rows) if rows is not None else None, n,
        _ptr(out), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("fdo_decode rejected its arguments")
    return out, lse
