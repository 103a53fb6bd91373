"""split_kv_gb300 -- split-KV decode attention (Flash-Decoding) for GB300.

A thin ctypes binding over the C ABI of ``lib/libfd.so`` (declared in
``include/fd.h``).  Every function has the C name and does argument
marshalling only: torch tensors are passed as device pointers, streams as
``cudaStream_t`` handles, and every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if the library is missing
the first call raises.

Typical use::

    import split_kv_gb300 as fd
    desc = fd.make_desc(q, k_cache, v_cache, max_seqlen=int(seqlens_host.max()))
    desc.n_splits = fd.fd_plan(B, Hq, Hkv, 128, seqlens_host)
    ws = torch.empty(fd.fd_workspace_size(desc, desc.n_splits), dtype=torch.uint8, device="cuda")
    fd.check(fd.fd_decode(desc, q, k_cache, v_cache, seqlens, None, out, lse, ws))
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import _build

FD_OK = 0
FD_ERR_INVALID_ARG = -1
FD_ERR_UNSUPPORTED = -2
FD_ERR_WORKSPACE = -3
FD_ERR_CUDA = -4
FD_ERR_DEVICE_TIMEOUT = -5
FD_ERR_DEVICE_BOUNDS = -6

FD_F16, FD_BF16, FD_F32, FD_E4M3 = 0, 1, 2, 3
FD_MAX_SPLITS = 128
FD_TILE_TOKENS = 128
FD_STATIC_WORKSPACE_BYTES = 8 << 20
FD_FLAG_CUDA_CORES = 1
FD_FLAG_TEST_DROP_FIRST_STAGE = 1 << 16

LIB_PATH = _build.LIB_PATH

# every function the header declares (checked against include/fd.h by the tests)
EXPORTS = ("fd_abi_version", "fd_status_string", "fd_num_sms", "fd_plan_splits", "fd_plan",
           "fd_plan_desc", "fd_workspace_size", "fd_decode", "fd_split_states", "fd_combine_states",
           "fd_device_status", "fd_decode_status", "fd_decode_static")


class FdDesc(ctypes.Structure):
    """Mirror of ``fd_desc`` (include/fd.h)."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("q_stride_b", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
        ("k_stride_b", ctypes.c_int64), ("k_stride_h", ctypes.c_int64), ("k_stride_t", ctypes.c_int64),
        ("v_stride_b", ctypes.c_int64), ("v_stride_h", ctypes.c_int64), ("v_stride_t", ctypes.c_int64),
        ("kv_extent", ctypes.c_int64),
        ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("max_seqlen", ctypes.c_int32), ("n_splits", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("q_len", ctypes.c_int32),
        ("q_stride_t", ctypes.c_int64),
        ("q_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]

    def copy(self) -> "FdDesc":
        d = FdDesc()
        ctypes.pointer(d)[0] = self
        return d


class FdError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {fd_status_string(status)} ({status})" if what
                         else f"{fd_status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                               "(the decode path has no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
        dp = ctypes.POINTER(FdDesc)
        sig = {
            "fd_abi_version": (i32, []),
            "fd_status_string": (ctypes.c_char_p, [i32]),
            "fd_num_sms": (i32, [i32]),
            "fd_plan_splits": (i32, [i64, i64, i64, i32]),
            "fd_plan": (i32, [i32, i32, i32, i32, vp, vp, i32, i32, i32]),
            "fd_plan_desc": (i32, [dp, vp, i32]),
            "fd_workspace_size": (sz, [dp, i32]),
            "fd_decode": (i32, [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "fd_split_states": (i32, [dp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "fd_combine_states": (i32, [dp, vp, sz, vp, vp, vp]),
            "fd_device_status": (i32, [vp, i32]),
            "fd_decode_status": (i32, [vp]),
            "fd_decode_static": (i32, [dp, vp, vp, vp, vp, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _ptr(x):
    """Device/host address of a torch tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def check(status: int, what: str = "") -> int:
    if int(status) < 0:
        raise FdError(status, what)
    return int(status)


# ---------------------------------------------------------------- C ABI
def fd_abi_version() -> int:
    return int(_load().fd_abi_version())


def fd_status_string(status: int) -> str:
    return _load().fd_status_string(int(status)).decode()


def fd_num_sms(device: int = -1) -> int:
    return int(_load().fd_num_sms(int(device)))


def fd_plan_splits(work_items: int, slots: int, n_kv_blocks: int, max_splits: int = FD_MAX_SPLITS) -> int:
    return int(_load().fd_plan_splits(int(work_items), int(slots), int(n_kv_blocks), int(max_splits)))


def _host_i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


def fd_plan(batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, seqlens_host,
            num_sms: int = 0, *, block_table_host=None, page_size: int = 0) -> int:
    """Split count for one decode step (16-bit cache, one query per sequence).
    block_table_host: optional host [batch, max_pages_per_seq] int32 table of
    a paged cache with `page_size`-token pages; validated, never changes the plan."""
    sl = _host_i32(seqlens_host)
    if sl.shape[0] < batch:
        raise ValueError("seqlens_host shorter than batch")
    bt_ptr, mp = None, 0
    if block_table_host is not None:
        bt = np.ascontiguousarray(np.asarray(block_table_host, dtype=np.int32))
        if bt.ndim != 2 or bt.shape[0] < batch:
            raise ValueError("block_table_host must be [batch, max_pages_per_seq]")
        mp = bt.shape[1]
        bt_ptr = bt.ctypes.data
    r = _load().fd_plan(int(batch), int(n_q_heads), int(n_kv_heads), int(head_dim),
                        sl.ctypes.data if batch > 0 else None, bt_ptr, int(page_size), int(mp),
                        int(num_sms))
    return int(r)


def fd_plan_desc(desc: FdDesc, seqlens_host, num_sms: int = 0) -> int:
    """The split count fd_decode plans for `desc` (n_splits <= 0) with these lengths."""
    sl = _host_i32(seqlens_host)
    if sl.shape[0] < desc.batch:
        raise ValueError("seqlens_host shorter than batch")
    return int(_load().fd_plan_desc(ctypes.byref(desc), sl.ctypes.data if desc.batch > 0 else None,
                                    int(num_sms)))


def fd_workspace_size(desc: FdDesc, n_splits: int = 0) -> int:
    return int(_load().fd_workspace_size(ctypes.byref(desc), int(n_splits)))


def fd_decode(desc: FdDesc, q, k_cache, v_cache, seqlens, block_table, out, lse, workspace,
              workspace_bytes: int | None = None, stream=None) -> int:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return int(_load().fd_decode(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 _ptr(seqlens), _ptr(block_table), _ptr(out), _ptr(lse),
                                 _ptr(workspace), int(wb), _stream(stream)))


def fd_split_states(desc: FdDesc, q, k_cache, v_cache, seqlens, block_table, workspace,
                    workspace_bytes: int | None = None, stream=None) -> int:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return int(_load().fd_split_states(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(seqlens), _ptr(block_table), _ptr(workspace),
                                       int(wb), _stream(stream)))


def fd_combine_states(desc: FdDesc, workspace, out, lse, workspace_bytes: int | None = None,
                      stream=None) -> int:
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return int(_load().fd_combine_states(ctypes.byref(desc), _ptr(workspace), int(wb), _ptr(out),
                                         _ptr(lse), _stream(stream)))


def fd_decode_static(desc: FdDesc, q, k_cache, v_cache, seqlens, block_table, out, lse,
                     stream=None) -> int:
    """fd_decode without a caller workspace: for callers that cannot allocate
    device memory; the states go to the library's fixed device array
    (FD_STATIC_WORKSPACE_BYTES per GPU; not used at all with one split).
    Calls that overlap on the GPU race on that array."""
    return int(_load().fd_decode_static(ctypes.byref(desc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(seqlens), _ptr(block_table), _ptr(out), _ptr(lse),
                                        _stream(stream)))


def fd_device_status(stream=None, clear: bool = True) -> int:
    return int(_load().fd_device_status(_stream(stream), 1 if clear else 0))


def fd_decode_status(stream=None) -> int:
    return int(_load().fd_decode_status(_stream(stream)))


# ---------------------------------------------------------------- helpers
def _dtype_code(t) -> int:
    import torch
    codes = {torch.float16: FD_F16, torch.bfloat16: FD_BF16, torch.float32: FD_F32}
    if hasattr(torch, "float8_e4m3fn"):
        codes[torch.float8_e4m3fn] = FD_E4M3
    return codes[t]


def make_desc(q, k_cache, v_cache, *, n_kv_heads: int | None = None, page_size: int = 0,
              max_pages_per_seq: int = 0, max_seqlen: int = 0, n_splits: int = 0,
              out_dtype=None, k_scale: float = 1.0, v_scale: float = 1.0) -> FdDesc:
    """Descriptor for q [B, Hq, D] (or a query block [B, q_len, Hq, D]) and a
    cache given as 4-D strided tensors: contiguous [B, Hkv, T, D] (page_size 0)
    or a paged pool [P, Hkv, page, D] (any strided view of that shape, e.g. a
    permuted [P, page, Hkv, D]).  An fp8 cache (torch.float8_e4m3fn) takes
    k_scale / v_scale: key = k_scale * stored, value = v_scale * stored."""
    import torch
    d = FdDesc()
    if q.dim() == 4:
        B, q_len, Hq, D = q.shape
        d.q_len = q_len
        d.q_stride_t = q.stride(1)
        d.q_stride_b, d.q_stride_h = q.stride(0), q.stride(2)
    else:
        B, Hq, D = q.shape
        d.q_len = 1
        d.q_stride_t = 0
        d.q_stride_b, d.q_stride_h = q.stride(0), q.stride(1)
    d.batch, d.n_q_heads, d.head_dim = B, Hq, D
    d.n_kv_heads = int(n_kv_heads if n_kv_heads is not None else k_cache.shape[1])
    d.kv_dtype = _dtype_code(k_cache.dtype)
    d.out_dtype = _dtype_code(out_dtype if out_dtype is not None else torch.float32)
    d.k_stride_b, d.k_stride_h, d.k_stride_t = k_cache.stride(0), k_cache.stride(1), k_cache.stride(2)
    d.v_stride_b, d.v_stride_h, d.v_stride_t = v_cache.stride(0), v_cache.stride(1), v_cache.stride(2)
    if page_size:
        d.kv_extent = k_cache.shape[0]
        d.page_size = page_size
        d.max_pages_per_seq = max_pages_per_seq
    else:
        d.kv_extent = k_cache.shape[2]
        d.page_size = 0
        d.max_pages_per_seq = 0
    d.max_seqlen = int(max_seqlen)
    d.n_splits = int(n_splits)
    d.flags = 0
    d.q_dtype = _dtype_code(q.dtype)
    d.reserved = 0
    d.k_scale, d.v_scale = float(k_scale), float(v_scale)
    return d
