"""Child process of tests/test_zz_no_alloc.py (not collected by pytest).

Runs fd_decode_static in two CUDA contexts of one device -- the primary
context and a second one created with the driver API -- and back in the
first, with every buffer allocated in the context that uses it and no torch
in the process.  The fixed array behind fd_decode_static lives once per
context, at an address that belongs to that context, so each call must find
its own context's copy.  Every result is checked against the oracle.  Prints
"ok" and exits 0 on success."""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import split_kv_gb300 as fd  # noqa: E402

ATOL, RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-3

cu = ctypes.CDLL("libcuda.so.1")


def ck(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what}: CUresult {rc}")


class Problem:
    """One fp16 decode step, n_splits = 3 (so the states go through the array)."""

    def __init__(self, seed):
        rng = np.random.default_rng(seed)
        self.B, self.Hq, self.Hkv, self.D, self.T = 2, 8, 2, 128, 1000
        self.q = rng.standard_normal((self.B, self.Hq, self.D)).astype(np.float16)
        self.k = rng.standard_normal((self.B, self.Hkv, self.T, self.D)).astype(np.float16)
        self.v = rng.standard_normal((self.B, self.Hkv, self.T, self.D)).astype(np.float16)
        self.sl = np.array([1000, 301], dtype=np.int32)
        self.ref_o, self.ref_l = oracle.decode(self.q, self.k, self.v, self.sl, dtype="f16",
                                               n_kv_heads=self.Hkv)

    def desc(self):
        d = fd.FdDesc()
        d.batch, d.n_q_heads, d.n_kv_heads, d.head_dim = self.B, self.Hq, self.Hkv, self.D
        d.kv_dtype, d.out_dtype, d.q_dtype = fd.FD_F16, fd.FD_F32, fd.FD_F16
        d.q_stride_b, d.q_stride_h = self.Hq * self.D, self.D
        d.k_stride_b, d.k_stride_h, d.k_stride_t = self.Hkv * self.T * self.D, self.T * self.D, self.D
        d.v_stride_b, d.v_stride_h, d.v_stride_t = d.k_stride_b, d.k_stride_h, d.k_stride_t
        d.kv_extent = self.T
        d.max_seqlen = int(self.sl.max())
        d.n_splits = 3
        d.q_len = 1
        d.k_scale = d.v_scale = 1.0
        return d


class DeviceBuffers:
    """The problem's inputs and outputs in the current context's memory."""

    def __init__(self, pb: Problem):
        self.ptrs = []
        self.q = self._upload(pb.q)
        self.k = self._upload(pb.k)
        self.v = self._upload(pb.v)
        self.sl = self._upload(pb.sl)
        self.n_out = pb.B * pb.Hq * pb.D
        self.out = self._alloc(4 * self.n_out)
        self.lse = self._alloc(4 * pb.B * pb.Hq)

    def _alloc(self, nbytes):
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
        self.ptrs.append(p.value)
        return p.value

    def _upload(self, a):
        a = np.ascontiguousarray(a)
        p = self._alloc(a.nbytes)
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), a.ctypes.data_as(ctypes.c_void_p),
                              ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")
        return p

    def download(self, p, shape):
        a = np.empty(shape, dtype=np.float32)
        ck(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(p),
                              ctypes.c_size_t(a.nbytes)), "cuMemcpyDtoH")
        return a


def run_and_check(pb: Problem, bufs: DeviceBuffers, what: str):
    # poison the outputs so that a call that writes nothing cannot pass
    nan = np.full(bufs.n_out, np.nan, dtype=np.float32)
    ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(bufs.out), nan.ctypes.data_as(ctypes.c_void_p),
                          ctypes.c_size_t(nan.nbytes)), "poison out")
    rc = fd.fd_decode_static(pb.desc(), bufs.q, bufs.k, bufs.v, bufs.sl, None, bufs.out, bufs.lse,
                             stream=0)
    if rc != fd.FD_OK:
        raise RuntimeError(f"{what}: fd_decode_static returned {rc}")
    ck(cu.cuCtxSynchronize(), f"{what}: synchronize")
    st = fd.fd_device_status(0, True)
    if st != fd.FD_OK:
        raise RuntimeError(f"{what}: device status {st}")
    o = bufs.download(bufs.out, (pb.B * pb.Hq, pb.D)).astype(np.float64)
    lse = bufs.download(bufs.lse, (pb.B * pb.Hq,)).astype(np.float64)
    err = np.abs(o - pb.ref_o)
    if not np.all(err <= ATOL + RTOL * np.abs(pb.ref_o)):
        raise RuntimeError(f"{what}: out differs from the oracle (max abs err {np.nanmax(err):.3e})")
    if not np.all(np.abs(lse - pb.ref_l) <= LSE_ATOL):
        raise RuntimeError(f"{what}: lse differs from the oracle")


def main():
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent(primary)")
    pb = Problem(71)
    in_primary = DeviceBuffers(pb)
    run_and_check(pb, in_primary, "primary context")

    second = ctypes.c_void_p()
    create = getattr(cu, "cuCtxCreate_v4", None)
    if create is not None:
        ck(create(ctypes.byref(second), None, 0, dev), "cuCtxCreate_v4")
    else:
        ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "cuCtxCreate_v2")
    ck(cu.cuCtxSetCurrent(second), "cuCtxSetCurrent(second)")
    in_second = DeviceBuffers(pb)
    run_and_check(pb, in_second, "second context")
    run_and_check(pb, in_second, "second context, again")

    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent(primary)")
    run_and_check(pb, in_primary, "primary context, after the second")
    print("ok")


if __name__ == "__main__":
    main()
