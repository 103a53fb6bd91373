"""The fused combine (FD_FLAG_FUSED_COMBINE): the last split CTA of each
(sequence, KV head, column block) group merges the group's rows, so a decode
step is one kernel.  It uses the combine kernel's arithmetic, so its results
must equal the two-kernel path's bit for bit; it is also checked against the
oracle, and the workspace's ticket section must be back at zero after every
call (including one that timed out)."""
import numpy as np
import pytest
import torch

import fd_inputs
import split_kv_gb300 as fd
from gpu_util import assert_parity, oracle_all

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
FP8 = hasattr(torch, "float8_e4m3fn")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from split_kv_gb300 import _build
    _build.build()
    torch.cuda.set_device(DEV)
    fd.fd_device_status(clear=True)
    yield


def _tickets(ws):
    return ws[:fd.FD_TICKET_BYTES].view(torch.int32)


def _decode(desc, q, k, v, sl, bt, ws, fused, out_dtype=torch.float32, with_lse=True, flags=0):
    B, Hq, D = desc.batch, desc.n_q_heads, desc.head_dim
    ql = max(1, desc.q_len)
    d = desc.copy() if hasattr(desc, "copy") else desc
    d.flags = flags | (fd.FD_FLAG_FUSED_COMBINE if fused else 0)
    d.out_dtype = {torch.float32: fd.FD_F32, torch.float16: fd.FD_F16, torch.bfloat16: fd.FD_BF16}[out_dtype]
    out = torch.full((B, ql, Hq, D), float("nan"), dtype=out_dtype, device=DEV)
    lse = torch.full((B, ql, Hq), float("nan"), dtype=torch.float32, device=DEV) if with_lse else None
    fd.check(fd.fd_decode(d, q, k, v, sl, bt, out, lse, ws), "fd_decode")
    return out, lse


def _problem(kind):
    """(desc, q, k, v, seqlens_dev, seqlens_host, block_table, q_dtype, oracle kwargs)"""
    D = 128
    bt = None
    okw = {}
    if kind == "contiguous":
        B, Hq, Hkv, T = 3, 32, 8, 9000
        lens = [9000, 129, 0]
        q = fd_inputs.randn((B, Hq, D), "f16", 3001, device=DEV)
        k = fd_inputs.randn((B, Hkv, T, D), "f16", 3002, device=DEV)
        v = fd_inputs.randn((B, Hkv, T, D), "f16", 3003, device=DEV)
        desc = fd.make_desc(q, k, v, max_seqlen=max(lens))
        qd = "f16"
    elif kind == "paged_g8":
        B, Hq, Hkv, ps = 2, 64, 8, 16
        lens = [3000, 777]
        mp = -(-max(lens) // ps)
        n_pages = B * mp + 5
        k = fd_inputs.randn((n_pages, Hkv, ps, D), "bf16", 3011, device=DEV)
        v = fd_inputs.randn((n_pages, Hkv, ps, D), "bf16", 3012, device=DEV)
        bt_h = fd_inputs.page_permutation(3013, n_pages)[:B * mp].reshape(B, mp).copy()
        bt = torch.from_numpy(bt_h).to(DEV)
        q = fd_inputs.randn((B, Hq, D), "bf16", 3014, device=DEV)
        desc = fd.make_desc(q, k, v, page_size=ps, max_pages_per_seq=mp, max_seqlen=max(lens))
        qd = "bf16"
        okw = dict(page_size=ps, block_table=bt_h)
    elif kind in ("block_q4_g4", "block_q4_g8", "g16"):
        G, ql = {"block_q4_g4": (4, 4), "block_q4_g8": (8, 4), "g16": (16, 1)}[kind]
        B, Hkv, T = 2, 2, 2500
        Hq = Hkv * G
        lens = [2500, 3]
        k = fd_inputs.randn((B, Hkv, T, D), "f16", 3021, device=DEV)
        v = fd_inputs.randn((B, Hkv, T, D), "f16", 3022, device=DEV)
        q = fd_inputs.randn((B, ql, Hq, D) if ql > 1 else (B, Hq, D), "f16", 3023, device=DEV)
        desc = fd.make_desc(q, k, v, max_seqlen=max(lens))
        qd = "f16"
    elif kind in ("fp8_g4", "fp8_block"):
        B, Hkv, T = 2, 4, 4000
        G, ql = (4, 1) if kind == "fp8_g4" else (4, 3)
        Hq = Hkv * G
        lens = [4000, 1100]
        k = fd_inputs.randn_fp8((B, Hkv, T, D), 3031, device=DEV, gain=16.0)
        v = fd_inputs.randn_fp8((B, Hkv, T, D), 3032, device=DEV, gain=16.0)
        q = fd_inputs.randn((B, ql, Hq, D) if ql > 1 else (B, Hq, D), "bf16", 3033, device=DEV)
        desc = fd.make_desc(q, k, v, max_seqlen=max(lens), k_scale=1 / 16, v_scale=1 / 16)
        qd = "bf16"
        okw = dict(kv_dtype="e4m3", k_scale=1 / 16, v_scale=1 / 16)
    else:
        raise ValueError(kind)
    sl_h = np.array(lens, dtype=np.int32)
    return desc, q, k, v, torch.from_numpy(sl_h).to(DEV), sl_h, bt, qd, okw


def _workspace(desc, S):
    wsb = fd.fd_workspace_size(desc, S)
    ws = torch.full((wsb,), 0x5A, dtype=torch.uint8, device=DEV)   # garbage everywhere ...
    fd.check(fd.fd_workspace_init(ws), "fd_workspace_init")         # ... but the tickets
    return ws


KINDS = ["contiguous", "paged_g8", "block_q4_g4", "block_q4_g8", "g16"] + (["fp8_g4", "fp8_block"] if FP8 else [])


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n_splits", [0, 1, 7, 128])
def test_fused_equals_two_kernel_path_bitwise(kind, n_splits):
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem(kind)
    desc.n_splits = n_splits
    S = n_splits if n_splits > 0 else None
    ws = _workspace(desc, n_splits)
    o1, l1 = _decode(desc, q, k, v, sl, bt, ws, fused=False)
    assert int(_tickets(ws).abs().sum().item()) == 0       # the two-kernel path leaves them alone
    o2, l2 = _decode(desc, q, k, v, sl, bt, ws, fused=True)
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert int(_tickets(ws).abs().sum().item()) == 0       # every group's ticket back at 0
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32)), f"{kind} S={S}: out differs"
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32)), f"{kind} S={S}: lse differs"
    if n_splits in (0, 128):
        rows = o2.numel() // 128
        ref_o, ref_l = oracle_all(q, k, v, sl_h, qd, desc.n_kv_heads, **okw)
        assert_parity(o2.cpu().double().numpy().reshape(rows, 128), l2.cpu().double().numpy().reshape(-1),
                      ref_o, ref_l, f"fused {kind} S={S}")


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_fused_low_precision_outputs_and_no_lse(out_dtype):
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem("contiguous")
    ws = _workspace(desc, 0)
    o1, _ = _decode(desc, q, k, v, sl, bt, ws, fused=False, out_dtype=out_dtype, with_lse=False)
    o2, _ = _decode(desc, q, k, v, sl, bt, ws, fused=True, out_dtype=out_dtype, with_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert int(_tickets(ws).abs().sum().item()) == 0


def test_fused_cuda_core_consumer():
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem("contiguous")
    ws = _workspace(desc, 0)
    o1, l1 = _decode(desc, q, k, v, sl, bt, ws, fused=False, flags=fd.FD_FLAG_CUDA_CORES)
    o2, l2 = _decode(desc, q, k, v, sl, bt, ws, fused=True, flags=fd.FD_FLAG_CUDA_CORES)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_fused_reports_tickets_that_were_not_zeroed():
    """A workspace whose ticket section holds garbage: the call records
    FD_ERR_WORKSPACE in the status word; after fd_workspace_init the next
    call is correct and leaves the tickets at zero."""
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem("contiguous")
    wsb = fd.fd_workspace_size(desc, 0)
    ws = torch.full((wsb,), 0x5A, dtype=torch.uint8, device=DEV)   # never initialised
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    _decode(desc, q, k, v, sl, bt, ws, fused=True)
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_WORKSPACE
    fd.check(fd.fd_workspace_init(ws))
    o2, l2 = _decode(desc, q, k, v, sl, bt, ws, fused=True)
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert int(_tickets(ws).abs().sum().item()) == 0
    ref_o, ref_l = oracle_all(q, k, v, sl_h, qd, desc.n_kv_heads)
    assert_parity(o2.cpu().double().numpy().reshape(-1, 128), l2.cpu().double().numpy().reshape(-1),
                  ref_o, ref_l, "fused after init")


def test_fused_workspace_serves_any_later_shape():
    """One initialisation: fused and two-kernel calls of different shapes
    alternate on the same workspace, and every fused call stays correct."""
    wsb = max(fd.fd_workspace_size(_problem(k)[0], 128) for k in ("contiguous", "block_q4_g8"))
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    fd.check(fd.fd_workspace_init(ws))
    for kind, S in (("contiguous", 128), ("block_q4_g8", 0), ("paged_g8", 3), ("contiguous", 0)):
        desc, q, k, v, sl, sl_h, bt, qd, okw = _problem(kind)
        desc.n_splits = S
        o1, l1 = _decode(desc, q, k, v, sl, bt, ws, fused=False)
        o2, l2 = _decode(desc, q, k, v, sl, bt, ws, fused=True)
        torch.cuda.synchronize()
        assert fd.fd_device_status(clear=True) == fd.FD_OK
        assert torch.equal(o1.view(torch.int32), o2.view(torch.int32)), kind
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32)), kind


def test_fused_replays_from_a_cuda_graph():
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem("contiguous")
    desc.n_splits = fd.fd_plan(desc.batch, desc.n_q_heads, desc.n_kv_heads, 128, sl_h)
    desc.flags = fd.FD_FLAG_FUSED_COMBINE
    ws = _workspace(desc, desc.n_splits)
    out = torch.empty(desc.batch, desc.n_q_heads, 128, dtype=torch.float32, device=DEV)
    lse = torch.empty(desc.batch, desc.n_q_heads, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode(desc, q, k, v, sl, None, out, lse, ws))
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fd.check(fd.fd_decode(desc, q, k, v, sl, None, out, lse, ws, stream=cap))
    for rep in range(4):
        q.copy_(fd_inputs.randn(tuple(q.shape), "f16", 3100 + rep, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_all(q, k, v, sl_h, qd, desc.n_kv_heads)
        assert_parity(out.cpu().double().numpy().reshape(-1, 128), lse.cpu().double().numpy().reshape(-1),
                      ref_o, ref_l, f"fused graph replay {rep}")
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert int(_tickets(ws).abs().sum().item()) == 0


def test_fused_static_entry_point():
    desc, q, k, v, sl, sl_h, bt, qd, okw = _problem("paged_g8")
    ws = _workspace(desc, 0)
    o1, l1 = _decode(desc, q, k, v, sl, bt, ws, fused=True)
    d = desc
    d.flags = fd.FD_FLAG_FUSED_COMBINE
    o2 = torch.full_like(o1, float("nan"))
    l2 = torch.full_like(l1, float("nan"))
    fd.check(fd.fd_decode_static(d, q, k, v, sl, bt, o2, l2), "fd_decode_static")
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert torch.equal(o1.view(torch.int32), o2.view(torch.int32))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


def test_fused_timeout_leaves_tickets_zero():
    """A call whose first stage never arrives: the bounded wait runs out, the
    status word reports the timeout, the CTAs that gave up still take their
    tickets (so the section is back at zero) and the next call is correct."""
    import time
    B, Hq, Hkv, D, T = 1, 8, 8, 128, 300
    q = fd_inputs.randn((B, Hq, D), "f16", 3201, device=DEV)
    k = fd_inputs.randn((B, Hkv, T, D), "f16", 3202, device=DEV)
    v = fd_inputs.randn((B, Hkv, T, D), "f16", 3203, device=DEV)
    sl_h = np.array([T], dtype=np.int32)
    sl = torch.from_numpy(sl_h).to(DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=T, n_splits=2)
    ws = _workspace(desc, 2)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    t0 = time.time()
    _decode(desc, q, k, v, sl, None, ws, fused=True, flags=fd.FD_FLAG_TEST_DROP_FIRST_STAGE)
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    assert int(_tickets(ws).abs().sum().item()) == 0
    o2, l2 = _decode(desc, q, k, v, sl, None, ws, fused=True)
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    ref_o, ref_l = oracle_all(q, k, v, sl_h, "f16", Hkv)
    assert_parity(o2.cpu().double().numpy().reshape(-1, 128), l2.cpu().double().numpy().reshape(-1),
                  ref_o, ref_l, "fused after a timeout")
