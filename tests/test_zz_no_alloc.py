"""fd_decode_static: the entry point for callers that cannot allocate device
memory (custom allocators that must not be re-entered, embedders that forbid
allocation after start-up, runtimes that own all device memory).  It keeps
the split states in the library's fixed device array instead of a caller
workspace.  Checked through the C ABI against fd_decode on two calls in a
row (different problems, so the second call runs over what the first left in
the shared array), plus the size limit.

This file is named to be collected last; it also passes alone in a fresh
process (it builds and loads the library itself)."""
import numpy as np
import pytest
import torch

import fd_inputs
import split_kv_gb300 as fd
from gpu_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    fd.fd_device_status(clear=True)
    yield


def _problem(B, Hq, Hkv, T, lens, dtype, seed, page_size=0):
    D = 128
    q = fd_inputs.randn((B, Hq, D), dtype, seed, device=DEV)
    sl_h = np.asarray(lens, dtype=np.int32)
    if page_size:
        mp = -(-T // page_size)
        n_pages = B * mp
        k = fd_inputs.randn((n_pages, Hkv, page_size, D), dtype, seed + 1, device=DEV)
        v = fd_inputs.randn((n_pages, Hkv, page_size, D), dtype, seed + 2, device=DEV)
        bt = torch.from_numpy(fd_inputs.block_table(seed + 3, B, mp, n_pages)).to(DEV)
        desc = fd.make_desc(q, k, v, page_size=page_size, max_pages_per_seq=mp,
                            max_seqlen=int(sl_h.max()))
    else:
        k = fd_inputs.randn((B, Hkv, T, D), dtype, seed + 1, device=DEV)
        v = fd_inputs.randn((B, Hkv, T, D), dtype, seed + 2, device=DEV)
        bt = None
        desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()))
    return desc, q, k, v, torch.from_numpy(sl_h).to(DEV), bt


def _with_workspace(desc, q, k, v, sl, bt):
    B, Hq, D = q.shape
    wsb = fd.fd_workspace_size(desc, 0)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode(desc, q, k, v, sl, bt, out, lse, ws), "fd_decode")
    return out, lse


def _static(desc, q, k, v, sl, bt):
    B, Hq, D = q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode_static(desc, q, k, v, sl, bt, out, lse), "fd_decode_static")
    return out, lse


def test_static_workspace_matches_fd_decode_two_calls_in_a_row():
    # two different problems back to back: the second reuses the array the
    # first one filled (more rows x splits in the first, fewer in the second)
    probs = [
        _problem(3, 32, 8, 9000, [9000, 129, 0], "f16", 41),
        _problem(2, 16, 2, 4096, [4096, 777], "bf16", 42, page_size=16),
    ]
    for desc, q, k, v, sl, bt in probs:
        want_o, want_l = _with_workspace(desc, q, k, v, sl, bt)
        got_o, got_l = _static(desc, q, k, v, sl, bt)
        torch.cuda.synchronize()
        assert fd.fd_device_status(clear=True) == fd.FD_OK
        B, Hq, D = q.shape
        assert_parity(got_o.cpu().double().numpy().reshape(B * Hq, D),
                      got_l.cpu().double().numpy().reshape(-1),
                      want_o.cpu().double().numpy().reshape(B * Hq, D),
                      want_l.cpu().double().numpy().reshape(-1), "fd_decode_static")


def test_static_workspace_rejects_problems_beyond_its_size():
    # 128 sequences x 32 query heads x 8 splits needs ~16.6 MiB of states
    desc, q, k, v, sl, bt = _problem(128, 32, 8, 64, [64] * 128, "f16", 43)
    desc.n_splits = 8
    assert fd.fd_workspace_size(desc, 8) > fd.FD_STATIC_WORKSPACE_BYTES
    out = torch.zeros(128, 32, 128, dtype=torch.float32, device=DEV)
    assert fd.fd_decode_static(desc, q, k, v, sl, bt, out, None) == fd.FD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0      # nothing was enqueued
