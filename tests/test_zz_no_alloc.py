"""fd_decode_static: the entry point for callers that cannot allocate device
memory (custom allocators that must not be re-entered, embedders that forbid
allocation after start-up, runtimes that own all device memory).  It keeps
the split states in the library's fixed device array instead of a caller
workspace.

Checked through the C ABI, on two calls in a row each time (different
problems, so the second call runs over what the first left in the shared
array): against the oracle element by element and against fd_decode, for a
16-bit cache, a paged cache, an fp8 (E4M3) cache and a query block on the
tcgen05 kernel.  Also: the size limit, the one-split case that needs no array,
no device memory allocated by a call, and the array found again in a second
CUDA context of the same device.

This file is named to be collected last; it also passes alone in a fresh
process (it builds and loads the library itself)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import fd_inputs
import split_kv_gb300 as fd
from gpu_util import assert_parity, oracle_all

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    fd.fd_device_status(clear=True)
    yield


def _problem(B, Hq, Hkv, T, lens, dtype, seed, page_size=0, q_len=1, fp8=False):
    """(desc, q, k, v, seqlens, block table, oracle kwargs) of one problem."""
    D = 128
    qshape = (B, q_len, Hq, D) if q_len > 1 else (B, Hq, D)
    q = fd_inputs.randn(qshape, dtype, seed, device=DEV)
    sl_h = np.asarray(lens, dtype=np.int32)
    okw = dict(dtype=dtype, n_kv_heads=Hkv)
    if page_size:
        mp = -(-T // page_size)
        n_pages = B * mp
        k = fd_inputs.randn((n_pages, Hkv, page_size, D), dtype, seed + 1, device=DEV)
        v = fd_inputs.randn((n_pages, Hkv, page_size, D), dtype, seed + 2, device=DEV)
        bt_h = fd_inputs.block_table(seed + 3, B, mp, n_pages)
        bt = torch.from_numpy(bt_h).to(DEV)
        desc = fd.make_desc(q, k, v, page_size=page_size, max_pages_per_seq=mp,
                            max_seqlen=int(sl_h.max()))
        okw.update(page_size=page_size, block_table=bt_h)
    elif fp8:
        k = fd_inputs.randn_fp8((B, Hkv, T, D), seed + 1, device=DEV, gain=16.0)
        v = fd_inputs.randn_fp8((B, Hkv, T, D), seed + 2, device=DEV, gain=16.0)
        bt = None
        desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()), k_scale=1 / 16, v_scale=1 / 16)
        okw.update(kv_dtype="e4m3", k_scale=1 / 16, v_scale=1 / 16)
    else:
        k = fd_inputs.randn((B, Hkv, T, D), dtype, seed + 1, device=DEV)
        v = fd_inputs.randn((B, Hkv, T, D), dtype, seed + 2, device=DEV)
        bt = None
        desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()))
    return desc, q, k, v, torch.from_numpy(sl_h).to(DEV), bt, okw


def _rows(q):
    return q.shape[0] * (q.shape[1] if q.dim() == 4 else 1) * q.shape[-2]


def _with_workspace(desc, q, k, v, sl, bt):
    wsb = fd.fd_workspace_size(desc, 0)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty(_rows(q), 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(_rows(q), dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode(desc, q, k, v, sl, bt, out, lse, ws), "fd_decode")
    return out, lse


def _static(desc, q, k, v, sl, bt, out=None, lse=None):
    if out is None:
        out = torch.full((_rows(q), 128), float("nan"), dtype=torch.float32, device=DEV)
        lse = torch.full((_rows(q),), float("nan"), dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode_static(desc, q, k, v, sl, bt, out, lse), "fd_decode_static")
    return out, lse


def _np(t):
    return t.cpu().double().numpy()


def _check_two_in_a_row(probs):
    """Each problem through fd_decode_static, one after the other: against the
    oracle, and against fd_decode on the same inputs."""
    for desc, q, k, v, sl, bt, okw in probs:
        got_o, got_l = _static(desc, q, k, v, sl, bt)
        want_o, want_l = _with_workspace(desc, q, k, v, sl, bt)
        torch.cuda.synchronize()
        assert fd.fd_device_status(clear=True) == fd.FD_OK
        ref_o, ref_l = oracle_all(q, k, v, sl.cpu().numpy(), **okw)
        S = fd.fd_plan_desc(desc, sl.cpu().numpy())
        what = f"fd_decode_static S={S}"
        assert S > 1          # the states go through the array
        assert_parity(_np(got_o), _np(got_l), ref_o, ref_l, what + " vs oracle")
        assert_parity(_np(got_o), _np(got_l), _np(want_o), _np(want_l), what + " vs fd_decode")


def test_static_workspace_matches_oracle_and_fd_decode_two_calls_in_a_row():
    # more rows x splits in the first problem, fewer in the second
    _check_two_in_a_row([
        _problem(3, 32, 8, 9000, [9000, 129, 0], "f16", 41),
        _problem(2, 16, 2, 4096, [4096, 777], "bf16", 42, page_size=16),
    ])


def test_static_workspace_fp8_cache_and_query_block_two_calls_in_a_row():
    # an E4M3 cache (bf16 q), then a 4-position query block of 8 heads per KV
    # head (32 columns: the tcgen05 kernel)
    _check_two_in_a_row([
        _problem(2, 32, 8, 5000, [5000, 2049], "bf16", 44, fp8=True),
        _problem(2, 16, 2, 3000, [3000, 1111], "bf16", 45, q_len=4),
    ])


def test_static_workspace_rejects_problems_beyond_its_size():
    # 128 sequences x 32 query heads x 8 splits needs ~16.6 MiB of states
    desc, q, k, v, sl, bt, _ = _problem(128, 32, 8, 64, [64] * 128, "f16", 43)
    desc.n_splits = 8
    assert fd.fd_workspace_size(desc, 8) > fd.FD_STATIC_WORKSPACE_BYTES
    out = torch.zeros(128, 32, 128, dtype=torch.float32, device=DEV)
    assert fd.fd_decode_static(desc, q, k, v, sl, bt, out, None) == fd.FD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0      # nothing was enqueued


def test_static_one_split_needs_no_array():
    """With one split the kernel writes out and lse itself, so a problem whose
    states would not fit the array still runs (72 x 256 rows > 16131)."""
    desc, q, k, v, sl, bt, okw = _problem(72, 256, 8, 200, [200 - (b % 7) for b in range(72)],
                                          "bf16", 46)
    desc.n_splits = 1
    assert fd.fd_workspace_size(desc, 2) > fd.FD_STATIC_WORKSPACE_BYTES
    got_o, got_l = _static(desc, q, k, v, sl, bt)
    want_o, want_l = _with_workspace(desc, q, k, v, sl, bt)
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert torch.equal(got_o, want_o) and torch.equal(got_l, want_l)   # the same launch
    rows = np.random.default_rng(3).choice(_rows(q), size=96, replace=False)
    ref_o, ref_l = oracle_all(q, k, v, sl.cpu().numpy(), rows=rows, **okw)
    assert_parity(_np(got_o)[rows], _np(got_l)[rows], ref_o, ref_l, "fd_decode_static S=1")
    desc.n_splits = 2
    assert fd.fd_decode_static(desc, q, k, v, sl, bt, got_o, got_l) == fd.FD_ERR_WORKSPACE


def test_static_call_allocates_no_device_memory():
    """Free device memory is the same before and after a call (after a first
    call of the same kernels, which loads them): a problem of another size,
    planned and forced split counts, with and without a query block."""
    a = _problem(2, 32, 8, 3000, [3000, 17], "f16", 47)
    b = _problem(4, 32, 8, 7000, [7000, 6999, 1, 4000], "f16", 48)
    c = _problem(2, 16, 2, 2000, [2000, 33], "bf16", 49, q_len=4)
    d = _problem(3, 16, 2, 2500, [2500, 1, 2400], "bf16", 50, q_len=4)
    bufs = {}
    for name, (desc, q, k, v, sl, bt, _) in zip("abcd", (a, b, c, d)):
        bufs[name] = (torch.empty(_rows(q), 128, dtype=torch.float32, device=DEV),
                      torch.empty(_rows(q), dtype=torch.float32, device=DEV))
    for name in "ac":                       # first calls: the kernels get loaded
        desc, q, k, v, sl, bt, _ = (a if name == "a" else c)
        _static(desc, q, k, v, sl, bt, *bufs[name])
    torch.cuda.synchronize()
    for name, p in (("b", b), ("d", d)):
        desc, q, k, v, sl, bt, _ = p
        for S in (0, 5):
            desc.n_splits = S
            free0 = torch.cuda.mem_get_info(DEV)[0]
            _static(desc, q, k, v, sl, bt, *bufs[name])
            torch.cuda.synchronize()
            free1 = torch.cuda.mem_get_info(DEV)[0]
            assert free1 == free0, f"problem {name} S={S}: free memory {free0} -> {free1}"
    assert fd.fd_device_status(clear=True) == fd.FD_OK


def test_static_array_found_again_in_a_second_context():
    """The array has one address per CUDA context.  A torch-free child process
    calls fd_decode_static in the primary context, in a second context of the
    same device, and in the primary one again, checking each against the oracle."""
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "static_ctx_child.py")],
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
