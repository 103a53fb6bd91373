"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element by
element: |got - ref| <= 2e-3 + 1e-2 |ref| for out, |dlse| <= 1e-3, -inf exact.
Every written buffer is surrounded by canaries that must survive."""
import json
import math
import os

import numpy as np
import pytest
import torch

import fd_inputs
import oracle
import split_kv_gb300 as fd
from gpu_util import assert_parity, oracle_all, oracle_rows_contiguous, planned_splits, run_decode

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _build():
    from split_kv_gb300 import _build as b
    b.build()
    torch.cuda.set_device(DEV)
    fd.fd_device_status(clear=True)
    yield
    torch.cuda.synchronize()


def _cache(B, Hkv, T, D, dtype, seed, gain=1.0):
    k = fd_inputs.randn_chunked((B, Hkv, T, D), dtype, seed, device=DEV)
    v = fd_inputs.randn_chunked((B, Hkv, T, D), dtype, seed + 1, device=DEV)
    return k, v


# ---------------------------------------------------------------- tiny MHA
@pytest.mark.parametrize("n_splits", [0, 1, 3, 7, 128])
def test_tiny_mha_split_counts(n_splits):
    c = fd_inputs.WORKLOADS["tiny_mha"]
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"], device=DEV)
    k, v = _cache(B, Hkv, T, D, c["dtype"], c["seed"] + 10)
    sl = np.array([T], dtype=np.int32)
    got_o, got_l, S = run_decode(q, k, v, sl, n_splits=n_splits)
    ref_o, ref_l = oracle_all(q, k, v, sl, c["dtype"], Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, f"tiny_mha S={S}")
    if n_splits == 0:
        assert S == oracle.num_splits_ref(B * Hkv, 2 * fd.fd_num_sms(), -(-T // 128))


# ---------------------------------------------------------------- shapes
PATHS = [0, fd.FD_FLAG_CUDA_CORES]   # tensor-core consumer (default), CUDA-core consumer


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_group_sizes_and_dtypes(dtype, group, flags):
    B, Hkv, D, T = 2, 4, 128, 1500
    Hq = Hkv * group
    q = fd_inputs.randn((B, Hq, D), dtype, 100 + group, device=DEV)
    k, v = _cache(B, Hkv, T, D, dtype, 200 + group)
    sl = np.array([1500, 333], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl, dtype, Hkv)
    for S in (0, 5):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S, flags=flags)
        assert_parity(got_o, got_l, ref_o, ref_l, f"G={group} {dtype} S={S} flags={flags}")


@pytest.mark.parametrize("flags", PATHS)
def test_ragged_lengths_and_empty_splits(flags):
    """Lengths at every tile / stage edge, a length-1 and a length-0 sequence,
    and split counts that leave most splits empty ("Flash-Decoding ..." §8
    functional checks).  The cache past each length is NaN: nothing of it may
    reach the result."""
    lens = [0, 1, 2, 63, 64, 65, 127, 128, 129, 191, 255, 256, 257, 300, 1000, 1025]
    B, Hq, Hkv, D, T = len(lens), 8, 2, 128, 1100
    q = fd_inputs.randn((B, Hq, D), "f16", 301, device=DEV)
    k, v = _cache(B, Hkv, T, D, "f16", 302)
    sl = np.array(lens, dtype=np.int32)
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        v[b, :, L:] = float("nan")
    ref_o, ref_l = oracle_all(q, k, v, sl, "f16", Hkv)
    for S in (0, 1, 2, 3, 8, 9, 128):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S, flags=flags)
        assert_parity(got_o, got_l, ref_o, ref_l, f"ragged S={S}")
        # the empty sequence: zero output and LSE = -inf exactly
        assert np.all(got_o[:Hq] == 0.0) and np.all(np.isneginf(got_l[:Hq]))


@pytest.mark.parametrize("flags", PATHS)
def test_adversarial_large_scores(flags):
    """q scaled so that scores reach about +-80 and beyond: the max
    subtraction must hold in both kernels, no inf or NaN anywhere."""
    B, Hq, Hkv, D, T = 2, 16, 4, 128, 32768
    k, v = _cache(B, Hkv, T, D, "f16", 401)
    sl = np.array([T, 4099], dtype=np.int32)
    for gain in (18.0, 40.0):
        q = fd_inputs.randn((B, Hq, D), "f16", 402, device=DEV, gain=gain)
        s = torch.einsum("bhd,bgtd->bhgt", q.float(), k.float()) / math.sqrt(D)
        assert s.abs().max().item() > 75.0
        del s
        for S in (0, 1, 128):
            got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S, flags=flags)
            ref_o, ref_l = oracle_all(q, k, v, sl, "f16", Hkv)
            assert_parity(got_o, got_l, ref_o, ref_l, f"gain={gain} S={S}")
            assert np.all(np.isfinite(got_l))


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_low_precision_outputs(out_dtype):
    B, Hq, Hkv, D, T = 2, 8, 2, 128, 2000
    q = fd_inputs.randn((B, Hq, D), "bf16", 501, device=DEV)
    k, v = _cache(B, Hkv, T, D, "bf16", 502)
    sl = np.array([2000, 3], dtype=np.int32)
    got_o, got_l, _ = run_decode(q, k, v, sl, out_dtype=out_dtype)
    ref_o, ref_l = oracle_all(q, k, v, sl, "bf16", Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, f"out {out_dtype}")


def test_strided_cache_and_query():
    """Token-major storage [B, T, Hkv, D] seen as a [B, Hkv, T, D] view, and a
    query that is a slice of a wider tensor."""
    B, Hq, Hkv, D, T = 2, 16, 4, 128, 900
    k_bthd = fd_inputs.randn((B, T, Hkv, D), "f16", 601, device=DEV)
    v_bthd = fd_inputs.randn((B, T, Hkv, D), "f16", 602, device=DEV)
    k, v = k_bthd.permute(0, 2, 1, 3), v_bthd.permute(0, 2, 1, 3)
    q_wide = fd_inputs.randn((B, Hq, 2 * D), "f16", 603, device=DEV)
    q = q_wide[:, :, D:]
    sl = np.array([900, 77], dtype=np.int32)
    got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=4)
    ref_o, ref_l = oracle_all(q, k, v, sl, "f16", Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, "strided")


# ---------------------------------------------------------------- paged
def _paged_problem(B, Hkv, D, ps, lens, dtype, seed, layout="HND", spare=7):
    max_pages = max(1, -(-max(lens) // ps))
    n_pages = B * max_pages + spare
    if layout == "HND":
        pk = fd_inputs.randn((n_pages, Hkv, ps, D), dtype, seed, device=DEV)
        pv = fd_inputs.randn((n_pages, Hkv, ps, D), dtype, seed + 1, device=DEV)
    else:   # [P, page, Hkv, D] storage seen as [P, Hkv, page, D]
        pk = fd_inputs.randn((n_pages, ps, Hkv, D), dtype, seed, device=DEV).permute(0, 2, 1, 3)
        pv = fd_inputs.randn((n_pages, ps, Hkv, D), dtype, seed + 1, device=DEV).permute(0, 2, 1, 3)
    perm = fd_inputs.page_permutation(seed + 2, n_pages)
    bt = perm[:B * max_pages].reshape(B, max_pages).copy()
    return pk, pv, bt


@pytest.mark.parametrize("ps", [8, 16, 32, 64, 128, 256])
def test_paged_page_sizes(ps):
    """Paged pool with a shuffled block table; pages past each length are NaN."""
    B, Hkv, G, D = 3, 2, 8, 128
    Hq = Hkv * G
    lens = [3000, 17, 1025]
    pk, pv, bt = _paged_problem(B, Hkv, D, ps, lens, "bf16", 700 + ps)
    q = fd_inputs.randn((B, Hq, D), "bf16", 701, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    for b, L in enumerate(lens):          # poison every slot past the length
        last = L // ps
        if L % ps:
            pk[int(bt[b, last]), :, L % ps:] = float("nan")
            pv[int(bt[b, last]), :, L % ps:] = float("nan")
        for jp in range(-(-L // ps), bt.shape[1]):
            pk[int(bt[b, jp])] = float("nan")
            pv[int(bt[b, jp])] = float("nan")
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "bf16", Hkv, page_size=ps, block_table=bt)
    for S in (0, 3):
        got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt, n_splits=S)
        assert_parity(got_o, got_l, ref_o, ref_l, f"paged ps={ps} S={S}")


def test_paged_token_major_pool():
    B, Hkv, G, D, ps = 2, 4, 4, 128, 16
    lens = [2049, 500]
    pk, pv, bt = _paged_problem(B, Hkv, D, ps, lens, "f16", 750, layout="NHD")
    q = fd_inputs.randn((B, Hkv * G, D), "f16", 751, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "f16", Hkv, page_size=ps, block_table=bt)
    assert_parity(got_o, got_l, ref_o, ref_l, "paged NHD")


@pytest.mark.parametrize("ps", [16, 64])
def test_paged_identity_table_is_bitwise_contiguous(ps):
    """A pool holding the contiguous cache page by page, read through the
    identity table, gives the contiguous result bit for bit."""
    B, Hkv, G, D, T = 2, 4, 4, 128, 4096
    k, v = _cache(B, Hkv, T, D, "f16", 801)
    q = fd_inputs.randn((B, Hkv * G, D), "f16", 802, device=DEV)
    npp = T // ps
    pk = k.reshape(B, Hkv, npp, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, D).contiguous()
    pv = v.reshape(B, Hkv, npp, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, D).contiguous()
    bt = np.arange(B * npp, dtype=np.int32).reshape(B, npp)
    sl = np.array([4096, 2500], dtype=np.int32)
    o1, l1, _ = run_decode(q, k, v, sl, n_splits=6)
    o2, l2, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt, n_splits=6)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("group,q_len", [(8, 4), (16, 8)])
def test_tcgen05_bitwise_repeatable_and_paged_identity(group, q_len):
    """The tcgen05 kernels (32 and 128 columns): two runs agree bit for bit,
    and a pool holding the contiguous cache page by page, read through the
    identity table, gives the contiguous result bit for bit."""
    B, Hkv, D, T, ps = 2, 2, 128, 4096, 64
    k, v = _cache(B, Hkv, T, D, "bf16", 811)
    q = fd_inputs.randn((B, q_len, Hkv * group, D), "bf16", 812, device=DEV)
    npp = T // ps
    pk = k.reshape(B, Hkv, npp, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, D).contiguous()
    pv = v.reshape(B, Hkv, npp, ps, D).permute(0, 2, 1, 3, 4).reshape(B * npp, Hkv, ps, D).contiguous()
    bt = np.arange(B * npp, dtype=np.int32).reshape(B, npp)
    sl = np.array([4096, 2500], dtype=np.int32)
    o1, l1, _ = run_decode(q, k, v, sl, n_splits=6)
    o2, l2, _ = run_decode(q, k, v, sl, n_splits=6)
    o3, l3, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt, n_splits=6)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


# ---------------------------------------------------------------- determinism, halves
def test_bitwise_repeatable_and_halves_equal_whole():
    B, Hq, Hkv, D, T = 2, 32, 8, 128, 6000
    q = fd_inputs.randn((B, Hq, D), "f16", 901, device=DEV)
    k, v = _cache(B, Hkv, T, D, "f16", 902)
    sl = np.array([6000, 4321], dtype=np.int32)
    o1, l1, S = run_decode(q, k, v, sl)
    o2, l2, _ = run_decode(q, k, v, sl)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # fd_split_states + fd_combine_states == fd_decode, bit for bit
    seqlens = torch.from_numpy(sl).to(DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=6000, n_splits=S)
    wsb = fd.fd_workspace_size(desc, S)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_split_states(desc, q, k, v, seqlens, None, ws))
    fd.check(fd.fd_combine_states(desc, ws, out, lse))
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().double().numpy().reshape(-1, D), o1)
    assert np.array_equal(lse.cpu().double().numpy().reshape(-1), l1)


@pytest.mark.parametrize("kind", ["f16", "bf16_cuda_cores", "fp8_block", "bf16_g8_q4", "f16_g16_q8"])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_one_split_writes_the_result_directly(kind, out_dtype):
    """With one split fd_decode (and fd_decode_static) skip the combine: the
    split kernel writes out / lse itself.  The bits must be those of
    fd_split_states + fd_combine_states, including an empty row, and the
    workspace must be left untouched."""
    B, Hkv, D, T = 3, 2, 128, 1500
    lens = np.array([1500, 77, 0], dtype=np.int32)
    flags, sc = 0, {}
    if kind == "fp8_block":
        if not hasattr(torch, "float8_e4m3fn"):
            pytest.skip("torch without float8_e4m3fn")
        G, ql = 4, 3
        k = fd_inputs.randn_fp8((B, Hkv, T, D), 1951, device=DEV, gain=16.0)
        v = fd_inputs.randn_fp8((B, Hkv, T, D), 1952, device=DEV, gain=16.0)
        q = fd_inputs.randn((B, ql, Hkv * G, D), "bf16", 1953, device=DEV)
        sc = dict(k_scale=1 / 16, v_scale=1 / 16)
    elif kind in ("bf16_g8_q4", "f16_g16_q8"):   # the two tcgen05 kernels
        G, ql = (8, 4) if kind == "bf16_g8_q4" else (16, 8)
        dt = kind.split("_")[0]
        k, v = _cache(B, Hkv, T, D, dt, 1956)
        q = fd_inputs.randn((B, ql, Hkv * G, D), dt, 1957, device=DEV)
    else:
        G, ql = 4, 1
        dt = "f16" if kind == "f16" else "bf16"
        k, v = _cache(B, Hkv, T, D, dt, 1954)
        q = fd_inputs.randn((B, Hkv * G, D), dt, 1955, device=DEV)
        flags = fd.FD_FLAG_CUDA_CORES if "cuda_cores" in kind else 0
    Hq = Hkv * G
    seqlens = torch.from_numpy(lens).to(DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=int(lens.max()), n_splits=1, out_dtype=out_dtype, **sc)
    desc.flags = flags
    wsb = fd.fd_workspace_size(desc, 1)
    shape = (B, ql, Hq, D)
    results = []
    for mode in ("two_kernels", "decode", "static"):
        ws = torch.full((wsb,), 0x5A, dtype=torch.uint8, device=DEV)
        out = torch.full(shape, float("nan"), dtype=out_dtype, device=DEV)
        lse = torch.full((B, ql, Hq), float("nan"), dtype=torch.float32, device=DEV)
        if mode == "two_kernels":
            fd.check(fd.fd_split_states(desc, q, k, v, seqlens, None, ws))
            fd.check(fd.fd_combine_states(desc, ws, out, lse))
        elif mode == "decode":
            fd.check(fd.fd_decode(desc, q, k, v, seqlens, None, out, lse, ws))
        else:
            fd.check(fd.fd_decode_static(desc, q, k, v, seqlens, None, out, lse))
        torch.cuda.synchronize()
        if mode == "decode":   # the direct path does not touch the workspace
            assert bool((ws == 0x5A).all())
        results.append((out.view(torch.int16 if out_dtype != torch.float32 else torch.int32).clone(),
                        lse.view(torch.int32).clone()))
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    for o, l in results[1:]:
        assert torch.equal(o, results[0][0]) and torch.equal(l, results[0][1])
    lse0 = results[0][1].view(torch.float32).cpu().numpy().reshape(B, ql * Hq)
    assert np.all(np.isneginf(lse0[2]))          # the empty row


def _states_workspace(desc, S, m, l, u):
    """A workspace in the documented layout filled with caller states."""
    rows = desc.batch * desc.n_q_heads
    D = desc.head_dim
    r256 = lambda x: (x + 255) // 256 * 256
    off_m = r256(rows * S * D * 4)
    off_l = off_m + r256(rows * S * 4)
    wsb = fd.fd_workspace_size(desc, S)
    assert wsb >= off_l + rows * S * 4
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    ws[:rows * S * D * 4].view(torch.float32).copy_(torch.tensor(u, dtype=torch.float32).reshape(-1))
    ws[off_m:off_m + rows * S * 4].view(torch.float32).copy_(torch.tensor(m, dtype=torch.float32).reshape(-1))
    ws[off_l:off_l + rows * S * 4].view(torch.float32).copy_(torch.tensor(l, dtype=torch.float32).reshape(-1))
    return ws, wsb


def test_combine_merges_the_pages_worked_states(golden_dir):
    """fd_combine_states on caller-given states: the 4.9 worked example (A, B)
    and the merge-trap states; an all-empty row gives 0 / -inf."""
    g = json.load(open(os.path.join(golden_dir, "dkv_worked_example.json")))
    t = json.load(open(os.path.join(golden_dir, "fd_merge_trap.json")))
    D = 128
    q = torch.zeros(1, 3, D, dtype=torch.float16, device=DEV)
    k = torch.zeros(1, 3, 8, D, dtype=torch.float16, device=DEV)
    desc = fd.make_desc(q, k, k, n_kv_heads=3, n_splits=3)
    S = 3
    m = np.full((3, S), -np.inf)
    l = np.zeros((3, S))
    u = np.zeros((3, S, D))
    # row 0: states A and B of the worked example, plus an empty split
    m[0, :2] = [math.log(2), math.log(4)]
    l[0, :2] = [g["block_A"]["ell"], g["block_B"]["ell"]]
    u[0, 0, :] = g["block_A"]["u"]
    u[0, 1, :] = g["block_B"]["u"]
    # row 1: merge trap, normalised states (lse_i, 1, o_i)
    m[1, :] = t["lse"]
    l[1, :] = 1.0
    u[1, :, :2] = np.array(t["o"])
    # row 2: every split empty
    ws, wsb = _states_workspace(desc, S, m, l, u)
    out = torch.empty(3, D, dtype=torch.float32, device=DEV)
    lse = torch.empty(3, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_combine_states(desc, ws, out, lse, wsb))
    torch.cuda.synchronize()
    o, L = out.cpu().double().numpy(), lse.cpu().double().numpy()
    np.testing.assert_allclose(o[0], g["merged"]["output"], rtol=2e-6)
    assert L[0] == pytest.approx(math.log(10.0), abs=2e-6)
    np.testing.assert_allclose(o[1, :2], t["printed_stable_merge"], rtol=0, atol=2e-6)
    assert np.all(o[1, 2:] == 0.0)
    assert L[1] == pytest.approx(t["printed_merged_lse"], abs=2e-5)
    assert np.all(o[2] == 0.0) and np.isneginf(L[2])


# ---------------------------------------------------------------- device bounds checks
def test_out_of_range_lengths_and_pages_are_reported():
    """Lengths beyond the capacity and block-table entries outside the pool are
    clamped / read as zeros on the device and reported in the status word."""
    B, Hkv, G, D, ps = 2, 2, 4, 128, 16
    pk, pv, bt = _paged_problem(B, Hkv, D, ps, [256, 256], "f16", 951)
    q = fd_inputs.randn((B, Hkv * G, D), "f16", 952, device=DEV)
    seqlens = torch.tensor([256, 256], dtype=torch.int32, device=DEV)
    desc = fd.make_desc(q, pk, pv, page_size=ps, max_pages_per_seq=bt.shape[1], n_splits=2)
    wsb = fd.fd_workspace_size(desc, 2)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty(B, Hkv * G, D, dtype=torch.float32, device=DEV)
    bad_bt = bt.copy()
    bad_bt[1, 3] = pk.shape[0] + 5
    bt_dev = torch.from_numpy(bad_bt).to(DEV)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    fd.check(fd.fd_decode(desc, q, pk, pv, seqlens, bt_dev, out, None, ws))
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_DEVICE_BOUNDS
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    too_long = torch.tensor([256, 10_000], dtype=torch.int32, device=DEV)
    fd.check(fd.fd_decode(desc, q, pk, pv, too_long, torch.from_numpy(bt).to(DEV), out, None, ws))
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_DEVICE_BOUNDS
    assert not torch.isnan(out).any()


# ---------------------------------------------------------------- the workloads at full size
def test_varlen_b16_full():
    c = fd_inputs.WORKLOADS["varlen_b16"]
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    sl = fd_inputs.varlen_seqlens(c["seed"], B, T)
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"], device=DEV)
    k, v = _cache(B, Hkv, T, D, c["dtype"], c["seed"] + 10)
    got_o, got_l, S = run_decode(q, k, v, sl)
    ref_o, ref_l = oracle_all(q, k, v, sl, c["dtype"], Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, f"varlen S={S}")


def test_long_gqa_128k_one_layer():
    """The headline workload at full size, in the bench's launch configuration
    (planned split count), every query row against the oracle."""
    c = fd_inputs.WORKLOADS["long_gqa_128k"]
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"], device=DEV)
    k, v = _cache(B, Hkv, T, D, c["dtype"], c["seed"] + 10)
    sl = np.array([T], dtype=np.int32)
    got_o, got_l, S = run_decode(q, k, v, sl)
    assert S == fd.fd_plan(1, Hq, Hkv, D, sl)
    ref_o, ref_l = oracle_all(q, k, v, sl, c["dtype"], Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, f"long_gqa_128k S={S}")


def test_paged_b8_full_sampled_rows():
    c = fd_inputs.WORKLOADS["paged_b8"]
    B, Hq, Hkv, D, T, ps = (c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"],
                            c["page_size"])
    npp = T // ps
    n_pages = B * npp
    pk = fd_inputs.randn_chunked((n_pages, Hkv, ps, D), c["dtype"], c["seed"], device=DEV)
    pv = fd_inputs.randn_chunked((n_pages, Hkv, ps, D), c["dtype"], c["seed"] + 1, device=DEV)
    bt = fd_inputs.block_table(c["seed"] + 2, B, npp, n_pages)
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"] + 3, device=DEV)
    sl = np.full(B, T, dtype=np.int32)
    got_o, got_l, S = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt)
    # the decode contract's planner, given the host block table, plans the same
    assert S == fd.fd_plan(B, Hq, Hkv, D, sl, block_table_host=bt, page_size=ps)
    rows = np.random.default_rng(5).choice(B * Hq, size=64, replace=False)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, c["dtype"], Hkv, page_size=ps, block_table=bt, rows=rows)
    assert_parity(got_o[rows], got_l[rows], ref_o, ref_l, f"paged_b8 S={S}")


@pytest.mark.parametrize("name", ["query_block_q4", "query_block_g8_q4", "query_block_g8_q8",
                                  "query_block_g16_q8"])
def test_query_block_workloads_full_sampled_rows(name):
    """The query-block workloads at full size (B = 4, 32K tokens) in the
    bench's launch configuration (planned split count; warp MMAs at 16
    columns, the tcgen05 kernels at 32, 64 and 128), sampled rows against the
    oracle, every position of the block represented."""
    c = fd_inputs.WORKLOADS[name]
    B, Hq, Hkv, D, T, ql = (c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"],
                            c["q_len"])
    q = fd_inputs.randn((B, ql, Hq, D), c["dtype"], c["seed"], device=DEV)
    k, v = _cache(B, Hkv, T, D, c["dtype"], c["seed"] + 10)
    sl = np.full(B, T, dtype=np.int32)
    got_o, got_l, S = run_decode(q, k, v, sl)
    assert S == planned_splits(B, Hq, Hkv, ql, sl)
    rng = np.random.default_rng(31)
    rows = np.sort(np.concatenate([
        ((b * ql + i) * Hq + rng.integers(0, Hq, size=1)) for b in range(B) for i in range(ql)]).ravel())
    ref_o, ref_l = oracle_all(q, k, v, sl, c["dtype"], Hkv, rows=rows)
    assert_parity(got_o[rows], got_l[rows], ref_o, ref_l, f"{name} S={S}")


@pytest.mark.parametrize("batch", [1, 4, 16, 64])
def test_sweep_plans_and_sampled_rows(batch):
    c = fd_inputs.WORKLOADS["sweep"]
    Hq, Hkv, D = c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
    rng = np.random.default_rng(batch)
    for ctx in c["ctxs"]:
        sl = np.full(batch, ctx, dtype=np.int32)
        q = fd_inputs.randn((batch, Hq, D), "f16", c["seed"] + batch, device=DEV)
        k, v = _cache(batch, Hkv, ctx, D, "f16", c["seed"] + 7 * batch + ctx)
        got_o, got_l, S = run_decode(q, k, v, sl)
        assert S == oracle.num_splits_ref(batch * Hkv, 2 * fd.fd_num_sms(), -(-ctx // 128))
        n_rows = batch * Hq if batch * Hq * ctx <= 4 * 32 * 262144 else 16
        rows = np.sort(rng.choice(batch * Hq, size=min(n_rows, batch * Hq), replace=False))
        ref_o, ref_l = oracle_rows_contiguous(q, k, v, sl, rows, "f16")
        assert_parity(got_o[rows], got_l[rows], ref_o, ref_l, f"sweep B={batch} ctx={ctx} S={S}")
        del k, v
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- LSE chaining, bounded waits
def test_lse_chaining_two_halves_merged_externally():
    """Decode the two halves of each sequence separately, then merge the two
    returned (out, lse) states with fd_combine_states: the result must equal
    the one-pass decode and the oracle ("Flash-Decoding ..." §8: return LSE
    and merge two halves externally, which catches base and scale bugs)."""
    B, Hq, Hkv, D, T, half = 2, 16, 4, 128, 6000, 2048
    q = fd_inputs.randn((B, Hq, D), "bf16", 1101, device=DEV)
    k, v = _cache(B, Hkv, T, D, "bf16", 1102)
    sl = np.array([6000, 5000], dtype=np.int32)
    o_full, l_full, _ = run_decode(q, k, v, sl)
    o1, l1, _ = run_decode(q, k[:, :, :half], v[:, :, :half], np.array([half, half], dtype=np.int32))
    o2, l2, _ = run_decode(q, k[:, :, half:], v[:, :, half:], sl - half)
    rows = B * Hq
    m = np.stack([l1, l2], axis=1)                 # natural-log LSE as the state max
    ell = np.ones((rows, 2))
    u = np.stack([o1, o2], axis=1)
    desc = fd.make_desc(q, k, v, n_splits=2)
    ws, wsb = _states_workspace(desc, 2, m, ell, u)
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_combine_states(desc, ws, out, lse, wsb))
    torch.cuda.synchronize()
    got_o = out.cpu().double().numpy().reshape(rows, D)
    got_l = lse.cpu().double().numpy().reshape(-1)
    ref_o, ref_l = oracle_all(q, k, v, sl, "bf16", Hkv)
    assert_parity(got_o, got_l, ref_o, ref_l, "two halves merged")
    np.testing.assert_allclose(got_o, o_full, rtol=0, atol=2e-5)
    np.testing.assert_allclose(got_l, l_full, rtol=0, atol=2e-5)


@pytest.mark.parametrize("kind", ["f16", "e4m3", "e4m3_two_per_cta", "f16_g8_q4", "bf16_g16_q8"])
def test_bounded_wait_reports_timeout_and_the_context_survives(kind):
    """The test hook drops the first K/V stage: the kernel's bounded wait runs
    out, the status word reports FD_ERR_DEVICE_TIMEOUT, nothing faults, and
    the next call on the same context is correct.  The 16-bit consumer, the
    fp8 one (which waits for two stages per iteration; with 20 splits x 8
    heads, more CTAs than SMs, each CTA serves two splits), and both tcgen05
    kernels (32 and 128 columns), whose MMA thread gives up on the missing
    stage and frees its tensor memory."""
    import time
    if kind.startswith("e4m3") and not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    G, ql = {"f16_g8_q4": (8, 4), "bf16_g16_q8": (16, 8)}.get(kind, (1, 1))
    dt = "bf16" if kind.startswith("bf16") else "f16"
    S = 20 if kind == "e4m3_two_per_cta" else 1
    B, Hkv, D, T = 1, 8 if G == 1 else 2, 128, 300 * S
    if S > 1:
        sms = torch.cuda.get_device_properties(DEV).multi_processor_count
        assert sms < B * Hkv * S and -(-S // 2) * B * Hkv <= sms   # the two-split CTA's range
    Hq = Hkv * G
    q = fd_inputs.randn((B, ql, Hq, D) if ql > 1 else (B, Hq, D), dt, 1201, device=DEV)
    sc = {}
    if kind.startswith("e4m3"):
        k = fd_inputs.randn_fp8((B, Hkv, T, D), 1203, device=DEV, gain=16.0)
        v = fd_inputs.randn_fp8((B, Hkv, T, D), 1204, device=DEV, gain=16.0)
        sc = dict(k_scale=1 / 16, v_scale=1 / 16)
    else:
        k, v = _cache(B, Hkv, T, D, dt, 1202)
    sl_h = np.array([T], dtype=np.int32)
    seqlens = torch.from_numpy(sl_h).to(DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=T, n_splits=S, **sc)
    desc.flags = fd.FD_FLAG_TEST_DROP_FIRST_STAGE
    ws = torch.empty(fd.fd_workspace_size(desc, S), dtype=torch.uint8, device=DEV)
    out = torch.zeros(B, ql, Hq, D, dtype=torch.float32, device=DEV)
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    t0 = time.time()
    fd.check(fd.fd_decode(desc, q, k, v, seqlens, None, out, None, ws))
    assert fd.fd_device_status(clear=True) == fd.FD_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    got_o, got_l, _ = run_decode(q, k, v, sl_h, n_splits=1, **sc)
    ref_o, ref_l = oracle_all(q, k, v, sl_h, dt, Hkv, kv_dtype="e4m3" if kind.startswith("e4m3") else None,
                              **sc)
    assert_parity(got_o, got_l, ref_o, ref_l, f"after a timed-out call ({kind})")


def test_fd_decode_replays_from_a_cuda_graph():
    """fd_decode allocates and synchronises nothing, so it can be captured in
    a CUDA graph; replays after the inputs change in place are correct."""
    B, Hq, Hkv, D, T = 2, 32, 8, 128, 3000
    q = fd_inputs.randn((B, Hq, D), "f16", 1301, device=DEV)
    k, v = _cache(B, Hkv, T, D, "f16", 1302)
    sl_h = np.array([3000, 1234], dtype=np.int32)
    seqlens = torch.from_numpy(sl_h).to(DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=T)
    desc.n_splits = fd.fd_plan(B, Hq, Hkv, D, sl_h)
    wsb = fd.fd_workspace_size(desc, desc.n_splits)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    out = torch.empty(B, Hq, D, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode(desc, q, k, v, seqlens, None, out, lse, ws))   # eager warm-up
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fd.check(fd.fd_decode(desc, q, k, v, seqlens, None, out, lse, ws, stream=cap))
    for seed in (1303, 1304):
        q.copy_(fd_inputs.randn((B, Hq, D), "f16", seed, device=DEV))
        k.copy_(fd_inputs.randn((B, Hkv, T, D), "f16", seed + 10, device=DEV))
        g.replay()
        torch.cuda.synchronize()
        ref_o, ref_l = oracle_all(q, k, v, sl_h, "f16", Hkv)
        assert_parity(out.cpu().double().numpy().reshape(B * Hq, D),
                      lse.cpu().double().numpy().reshape(-1), ref_o, ref_l, f"graph replay {seed}")
    assert fd.fd_device_status(clear=True) == fd.FD_OK


@pytest.mark.parametrize("kind", ["f16", "e4m3"])
def test_lengths_written_by_the_kernel_before(kind):
    """The split kernels prefetch the first tokens of their split into L2
    ahead of their launch wait, from a length read without waiting.  Here a
    kernel just before each call in the stream writes new lengths (longer,
    shorter, empty), with no synchronisation in between; every result is
    checked against the oracle.  The fp8 case runs the two-split CTA."""
    if kind == "e4m3" and not FP8:
        pytest.skip("torch without float8_e4m3fn")
    B, Hq, Hkv, D, T, S = 2, 32, 8, 128, 4096, 10
    q = fd_inputs.randn((B, Hq, D), "f16", 1311, device=DEV)
    sc = {}
    if kind == "e4m3":
        k = fd_inputs.randn_fp8((B, Hkv, T, D), 1312, device=DEV, gain=GAIN_K)
        v = fd_inputs.randn_fp8((B, Hkv, T, D), 1313, device=DEV, gain=GAIN_V)
        sc = dict(k_scale=1 / GAIN_K, v_scale=1 / GAIN_V)
    else:
        k, v = _cache(B, Hkv, T, D, "f16", 1312)
    seqlens = torch.zeros(B, dtype=torch.int32, device=DEV)
    desc = fd.make_desc(q, k, v, max_seqlen=T, n_splits=S, **sc)
    ws = torch.empty(fd.fd_workspace_size(desc, S), dtype=torch.uint8, device=DEV)
    outs = []
    all_lens = ([4096, 100], [37, 4000], [2048, 2049], [0, 4096], [4096, 4096])
    for lens in all_lens:
        src = torch.tensor(lens, dtype=torch.int32, device=DEV)
        torch.add(src, 0, out=seqlens)            # a kernel writes the lengths
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=DEV)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=DEV)
        fd.check(fd.fd_decode(desc, q, k, v, seqlens, None, out, lse, ws), "fd_decode")
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    for lens, (out, lse) in zip(all_lens, outs):
        ref_o, ref_l = oracle_all(q, k, v, np.array(lens, dtype=np.int32), "f16", Hkv,
                                  kv_dtype="e4m3" if kind == "e4m3" else None, **sc)
        assert_parity(out.cpu().double().numpy().reshape(B * Hq, D), lse.cpu().double().numpy().reshape(-1),
                      ref_o, ref_l, f"lengths {lens} ({kind})")


# ---------------------------------------------------------------- query blocks, any group
@pytest.mark.parametrize("q_len", [2, 4, 8])
@pytest.mark.parametrize("group", [1, 3, 4, 8])
def test_query_blocks(q_len, group):
    """Short query blocks ("Flash-Decoding ..." §7): position i of a sequence
    with L keys sees the first L - q_len + 1 + i ([DKV] §06 per-query
    visibility).  G*q_len ranges from 2 to 64 columns (1 to 4 CTAs per split);
    the 5-token sequence leaves early positions of an 8-block without keys."""
    B, Hkv, D, T = 3, 2, 128, 1200
    Hq = Hkv * group
    q = fd_inputs.randn((B, q_len, Hq, D), "bf16", 1400 + 10 * q_len + group, device=DEV)
    k, v = _cache(B, Hkv, T, D, "bf16", 1500 + group)
    sl = np.array([1200, 130, 5], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl, "bf16", Hkv)
    for S in (0, 3, 128):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S)
        assert_parity(got_o, got_l, ref_o, ref_l, f"q_len={q_len} G={group} S={S}")


@pytest.mark.parametrize("group,q_len,dtype", [(12, 6, "bf16"), (5, 16, "f16"), (16, 8, "bf16"),
                                               (9, 16, "f16"), (16, 16, "bf16")])
def test_query_blocks_wide(group, q_len, dtype):
    """Query blocks of 72, 80 and 128 columns (one tcgen05 CTA serves a KV
    head's whole group) and of 144 and 256 columns (column blocks of 16),
    against the oracle; one sequence shorter than the block, and NaN in the
    cache past its length."""
    B, Hkv, D, T = 2, 2, 128, 900
    Hq = Hkv * group
    q = fd_inputs.randn((B, q_len, Hq, D), dtype, 1450 + 10 * q_len + group, device=DEV)
    k, v = _cache(B, Hkv, T, D, dtype, 1550 + group)
    sl = np.array([900, 11], dtype=np.int32)
    k[1, :, 11:] = float("nan")
    v[1, :, 11:] = float("nan")
    ref_o, ref_l = oracle_all(q, k, v, sl, dtype, Hkv)
    for S in (0, 1, 5):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S)
        assert_parity(got_o, got_l, ref_o, ref_l, f"q_len={q_len} G={group} S={S}")


@pytest.mark.parametrize("group,q_len", [(8, 4), (16, 8)])
def test_query_blocks_wide_large_scores(group, q_len):
    """Scores into the hundreds on the tcgen05 kernels (32 and 128 columns):
    the lazily moved running max (moved only when a stage's max exceeds it by
    more than 2^8) must keep every weight finite and the merge exact."""
    B, Hkv, D, T = 2, 2, 128, 4096
    Hq = Hkv * group
    k, v = _cache(B, Hkv, T, D, "bf16", 1650 + group)
    sl = np.array([4096, 700], dtype=np.int32)
    for gain in (18.0, 40.0):
        q = fd_inputs.randn((B, q_len, Hq, D), "bf16", 1660 + group, device=DEV, gain=gain)
        ref_o, ref_l = oracle_all(q, k, v, sl, "bf16", Hkv)
        for S in (0, 1, 6):
            got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S)
            assert_parity(got_o, got_l, ref_o, ref_l, f"G={group} q_len={q_len} gain={gain} S={S}")
            assert np.all(np.isfinite(got_l))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_combine_of_many_rows(out_dtype):
    """1024 query rows (a warp of the combine per row): 3 and 40 splits (past
    the first 32 a lane holds), an empty sequence and a short one, every
    output dtype, against the oracle."""
    B, Hkv, G, ql, D, T = 8, 2, 16, 4, 128, 700
    Hq = Hkv * G
    q = fd_inputs.randn((B, ql, Hq, D), "bf16", 1680, device=DEV)
    k, v = _cache(B, Hkv, T, D, "bf16", 1681)
    sl = np.array([700, 0, 5, 350, 699, 64, 1, 700], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl, "bf16", Hkv)
    if out_dtype != torch.float32:
        ref_o = torch.from_numpy(ref_o).to(out_dtype).double().numpy()
    for S in (3, 40):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S, out_dtype=out_dtype)
        assert_parity(got_o, got_l, ref_o, ref_l, f"1024 rows S={S} out={out_dtype}")
        assert np.all(got_o.reshape(B, -1)[1] == 0.0) and np.all(np.isneginf(got_l.reshape(B, -1)[1]))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_combine_of_many_rows_unaligned_output(out_dtype):
    """out carries only its element alignment: the many-rows combine writes
    an output one element past an aligned address correctly, and the element
    before it stays untouched."""
    B, Hkv, G, ql, D, T = 8, 2, 16, 4, 128, 700
    Hq = Hkv * G
    rows = B * ql * Hq
    q = fd_inputs.randn((B, ql, Hq, D), "bf16", 1690, device=DEV)
    k, v = _cache(B, Hkv, T, D, "bf16", 1691)
    sl_h = np.array([700, 0, 5, 350, 699, 64, 1, 700], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl_h, "bf16", Hkv)
    ref_o = torch.from_numpy(ref_o).to(out_dtype).double().numpy()
    S = 5
    desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()), n_splits=S, out_dtype=out_dtype)
    ws = torch.empty(fd.fd_workspace_size(desc, S), dtype=torch.uint8, device=DEV)
    backing = torch.full((rows * D + 1,), float("nan"), dtype=out_dtype, device=DEV)
    out = backing[1:]
    assert out.data_ptr() % 16 != 0
    lse = torch.empty(rows, dtype=torch.float32, device=DEV)
    fd.check(fd.fd_decode(desc, q, k, v, torch.from_numpy(sl_h).to(DEV), None, out, lse, ws), "fd_decode")
    torch.cuda.synchronize()
    assert fd.fd_device_status(clear=True) == fd.FD_OK
    assert torch.isnan(backing[0]).item()
    assert_parity(out.double().cpu().numpy().reshape(rows, D), lse.double().cpu().numpy(), ref_o, ref_l,
                  f"unaligned out {out_dtype}")


def test_query_block_wide_paged():
    """A paged 128-column block (G = 16, q_len = 8) on the tcgen05 path."""
    B, Hkv, G, D, ps, ql = 2, 2, 16, 128, 64, 8
    lens = [1500, 333]
    pk, pv, bt = _paged_problem(B, Hkv, D, ps, lens, "bf16", 1603)
    q = fd_inputs.randn((B, ql, Hkv * G, D), "bf16", 1604, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "bf16", Hkv, page_size=ps, block_table=bt)
    assert_parity(got_o, got_l, ref_o, ref_l, "paged wide query block")


def test_query_block_paged_and_strided():
    B, Hkv, G, D, ps, ql = 2, 4, 4, 128, 16, 4
    lens = [2049, 700]
    pk, pv, bt = _paged_problem(B, Hkv, D, ps, lens, "f16", 1601)
    wide = fd_inputs.randn((B, ql, Hkv * G, 2 * D), "f16", 1602, device=DEV)
    q = wide[..., :D]                                   # strided query block
    sl = np.array(lens, dtype=np.int32)
    got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "f16", Hkv, page_size=ps, block_table=bt)
    assert_parity(got_o, got_l, ref_o, ref_l, "paged query block")


@pytest.mark.parametrize("group,dtype", [(24, "f16"), (32, "bf16"), (64, "f16"), (128, "bf16")])
def test_large_groups_single_query(group, dtype):
    """One query per sequence with 24 to 128 query heads per KV head (MQA-like
    groups): the group's heads are the tcgen05 kernels' columns."""
    B, Hkv, D, T = 2, 1, 128, 1800
    Hq = Hkv * group
    q = fd_inputs.randn((B, Hq, D), dtype, 1720 + group, device=DEV)
    k, v = _cache(B, Hkv, T, D, dtype, 1730 + group)
    sl = np.array([1800, 37], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl, dtype, Hkv)
    for S in (0, 1, 4):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S)
        assert_parity(got_o, got_l, ref_o, ref_l, f"G={group} S={S}")


@pytest.mark.parametrize("group", [3, 5, 16])
def test_other_group_sizes_single_query(group):
    """Groups that are not powers of two, and a 16-wide group, on the
    tensor-core path (one or two N blocks of the MMA)."""
    B, Hkv, D, T = 2, 2, 128, 2500
    Hq = Hkv * group
    q = fd_inputs.randn((B, Hq, D), "f16", 1700 + group, device=DEV)
    k, v = _cache(B, Hkv, T, D, "f16", 1710 + group)
    sl = np.array([2500, 901], dtype=np.int32)
    ref_o, ref_l = oracle_all(q, k, v, sl, "f16", Hkv)
    for S in (0, 7):
        got_o, got_l, _ = run_decode(q, k, v, sl, n_splits=S)
        assert_parity(got_o, got_l, ref_o, ref_l, f"G={group} S={S}")


# ---------------------------------------------------------------- fp8 (E4M3) caches
FP8 = hasattr(torch, "float8_e4m3fn")
fp8_only = pytest.mark.skipif(not FP8, reason="torch without float8_e4m3fn")
GAIN_K, GAIN_V = 64.0, 16.0          # stored = value x gain, scale = 1 / gain


def _nan_past_lengths_fp8(t, lens):
    """E4M3 NaN (0x7f) in every cache slot past each sequence's length."""
    raw = t.view(torch.uint8)
    for b, L in enumerate(lens):
        raw[b, :, L:] = 0x7F


@fp8_only
@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("group", [1, 4, 8])
def test_fp8_cache(q_dtype, group):
    B, Hkv, D, T = 3, 2, 128, 2100
    Hq = Hkv * group
    q = fd_inputs.randn((B, Hq, D), q_dtype, 1800 + group, device=DEV)
    k8 = fd_inputs.randn_fp8((B, Hkv, T, D), 1810 + group, device=DEV, gain=GAIN_K)
    v8 = fd_inputs.randn_fp8((B, Hkv, T, D), 1820 + group, device=DEV, gain=GAIN_V)
    lens = [2100, 130, 1]
    _nan_past_lengths_fp8(k8, lens)
    _nan_past_lengths_fp8(v8, lens)
    sl = np.array(lens, dtype=np.int32)
    sc = dict(k_scale=1 / GAIN_K, v_scale=1 / GAIN_V)
    ref_o, ref_l = oracle_all(q, k8, v8, sl, q_dtype, Hkv, kv_dtype="e4m3", **sc)
    for S in (0, 3, 128):
        got_o, got_l, _ = run_decode(q, k8, v8, sl, n_splits=S, **sc)
        assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 q={q_dtype} G={group} S={S}")


@fp8_only
@pytest.mark.parametrize("S", [10, 11])
def test_fp8_two_splits_per_cta(S):
    """More fp8 splits than SMs, with the CTAs of two splits (ceil(S / 2) per
    sequence and KV head) in one wave, so each CTA serves two splits with its
    two halves of threads and shared memory; with an odd S the second half
    of each (sequence, KV head)'s last CTA has no split.
    Ragged lengths with NaN past them; every row against the oracle."""
    B, Hkv, G, D, T = 2, 8, 4, 128, 3000
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert sms < B * Hkv * S and -(-S // 2) * B * Hkv <= sms   # the two-split CTA's range
    q = fd_inputs.randn((B, Hkv * G, D), "bf16", 1840 + S, device=DEV)
    k8 = fd_inputs.randn_fp8((B, Hkv, T, D), 1850 + S, device=DEV, gain=GAIN_K)
    v8 = fd_inputs.randn_fp8((B, Hkv, T, D), 1860 + S, device=DEV, gain=GAIN_V)
    lens = [3000, 1777]
    _nan_past_lengths_fp8(k8, lens)
    _nan_past_lengths_fp8(v8, lens)
    sl = np.array(lens, dtype=np.int32)
    sc = dict(k_scale=1 / GAIN_K, v_scale=1 / GAIN_V)
    ref_o, ref_l = oracle_all(q, k8, v8, sl, "bf16", Hkv, kv_dtype="e4m3", **sc)
    got_o, got_l, _ = run_decode(q, k8, v8, sl, n_splits=S, **sc)
    assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 two splits per CTA S={S}")


@fp8_only
@pytest.mark.parametrize("ps", [16, 64])
def test_fp8_paged_two_splits_per_cta(ps):
    """An fp8 pool through a shuffled block table with more CTAs than SMs
    (2 x 8 heads x 13 splits), so each CTA serves two splits, the second
    half of each (sequence, head)'s last CTA idle."""
    B, Hkv, G, D, S = 2, 8, 4, 128, 13
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    assert sms < B * Hkv * S and -(-S // 2) * B * Hkv <= sms   # the two-split CTA's range
    lens = [2600, 1333]
    max_pages = -(-max(lens) // ps)
    n_pages = B * max_pages + 5
    pk = fd_inputs.randn_fp8((n_pages, Hkv, ps, D), 1960 + ps, device=DEV, gain=GAIN_K)
    pv = fd_inputs.randn_fp8((n_pages, Hkv, ps, D), 1961 + ps, device=DEV, gain=GAIN_V)
    bt = fd_inputs.page_permutation(1962 + ps, n_pages)[:B * max_pages].reshape(B, max_pages).copy()
    q = fd_inputs.randn((B, Hkv * G, D), "bf16", 1963 + ps, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    sc = dict(k_scale=1 / GAIN_K, v_scale=1 / GAIN_V)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "bf16", Hkv, page_size=ps, block_table=bt,
                              kv_dtype="e4m3", **sc)
    got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt, n_splits=S, **sc)
    assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 paged two splits per CTA ps={ps}")


@fp8_only
@pytest.mark.parametrize("ps", [16, 64])
def test_fp8_paged_and_query_block(ps):
    """An fp8 pool read through a shuffled block table, with a 4-position
    query block of a G = 4 group (16 columns: two MMA N blocks)."""
    B, Hkv, G, D, ql = 2, 2, 4, 128, 4
    lens = [1500, 300]
    max_pages = -(-max(lens) // ps)
    n_pages = B * max_pages + 3
    pk = fd_inputs.randn_fp8((n_pages, Hkv, ps, D), 1900 + ps, device=DEV, gain=GAIN_K)
    pv = fd_inputs.randn_fp8((n_pages, Hkv, ps, D), 1901 + ps, device=DEV, gain=GAIN_V)
    bt = fd_inputs.page_permutation(1902 + ps, n_pages)[:B * max_pages].reshape(B, max_pages).copy()
    q = fd_inputs.randn((B, ql, Hkv * G, D), "f16", 1903, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    sc = dict(k_scale=1 / GAIN_K, v_scale=1 / GAIN_V)
    ref_o, ref_l = oracle_all(q, pk, pv, sl, "f16", Hkv, page_size=ps, block_table=bt,
                              kv_dtype="e4m3", **sc)
    for S in (0, 5):
        got_o, got_l, _ = run_decode(q, pk, pv, sl, page_size=ps, block_table=bt, n_splits=S, **sc)
        assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 paged ps={ps} S={S}")


@fp8_only
def test_fp8_long_gqa_128k_one_layer():
    c = fd_inputs.WORKLOADS["long_gqa_128k_fp8"]
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    g = c["kv_gain"]
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"], device=DEV)
    k8 = fd_inputs.randn_fp8((B, Hkv, T, D), c["seed"] + 10, device=DEV, gain=g)
    v8 = fd_inputs.randn_fp8((B, Hkv, T, D), c["seed"] + 11, device=DEV, gain=g)
    sl = np.array([T], dtype=np.int32)
    got_o, got_l, S = run_decode(q, k8, v8, sl, k_scale=1 / g, v_scale=1 / g)
    ref_o, ref_l = oracle_all(q, k8, v8, sl, c["dtype"], Hkv, kv_dtype="e4m3",
                              k_scale=1 / g, v_scale=1 / g)
    assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 long_gqa_128k S={S}")


@fp8_only
@pytest.mark.parametrize("q_dtype", ["f16", "bf16"])
def test_fp8_every_finite_code(q_dtype):
    """Every finite E4M3 pattern (254 of them: both zeros, subnormals, +-448)
    occurs in K and in V, so each one goes through the kernel's conversion;
    a ragged length puts NaN patterns in the tail that must stay unseen."""
    B, Hkv, G, D, T = 1, 1, 8, 128, 1016
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    rng = np.random.default_rng(2100)
    cells = T * D
    k_raw = rng.permutation(np.resize(codes, cells)).reshape(B, Hkv, T, D)
    v_raw = rng.permutation(np.resize(codes, cells)).reshape(B, Hkv, T, D)
    k8 = torch.from_numpy(k_raw.copy()).view(torch.float8_e4m3fn).to(DEV)
    v8 = torch.from_numpy(v_raw.copy()).view(torch.float8_e4m3fn).to(DEV)
    lens = [1001]
    _nan_past_lengths_fp8(k8, lens)
    _nan_past_lengths_fp8(v8, lens)
    q = fd_inputs.randn((B, Hkv * G, D), q_dtype, 2101, device=DEV)
    sl = np.array(lens, dtype=np.int32)
    sc = dict(k_scale=1 / 64, v_scale=1 / 64)
    ref_o, ref_l = oracle_all(q, k8, v8, sl, q_dtype, Hkv, kv_dtype="e4m3", **sc)
    for S in (0, 4):
        got_o, got_l, _ = run_decode(q, k8, v8, sl, n_splits=S, **sc)
        assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 every code q={q_dtype} S={S}")


@fp8_only
@pytest.mark.parametrize("case", ["small", "large"])
def test_fp8_bf16_query_magnitudes(case):
    """bf16 query heads of very different magnitudes against an fp8 cache:
    a zero head, heads near the bottom of the bf16 range, heads far above the
    f16 range (with a tiny k_scale so that their scores stay moderate), and a
    head whose dims differ by 2^20 among themselves."""
    B, Hkv, G, D, T = 2, 2, 4, 128, 1500
    Hq = Hkv * G
    base = fd_inputs.randn((B, Hq, D), "f32", 2200, device="cpu")
    if case == "small":
        heads = [1.0, 2.0 ** -8, 2.0 ** 4, 0.0, 2.0 ** -120, None, 2.0 ** -30, 1.0]
        k_scale = 1 / GAIN_K
    else:
        heads = [2.0 ** 20, 2.0 ** 16, 2.0 ** 18, 1.0, 2.0 ** 20, None, 2.0 ** -4, 2.0 ** 19]
        k_scale = 2.0 ** -20 / GAIN_K
    for h, f in enumerate(heads):
        if f is None:                    # dims 64.. are 2^-20 of dims ..63
            base[:, h, 64:] *= 2.0 ** -20
        else:
            base[:, h] *= f
    q = base.to(torch.bfloat16).to(DEV)
    k8 = fd_inputs.randn_fp8((B, Hkv, T, D), 2210, device=DEV, gain=GAIN_K)
    v8 = fd_inputs.randn_fp8((B, Hkv, T, D), 2211, device=DEV, gain=GAIN_V)
    sl = np.array([1500, 777], dtype=np.int32)
    sc = dict(k_scale=k_scale, v_scale=1 / GAIN_V)
    ref_o, ref_l = oracle_all(q, k8, v8, sl, "bf16", Hkv, kv_dtype="e4m3", **sc)
    for S in (0, 6):
        got_o, got_l, _ = run_decode(q, k8, v8, sl, n_splits=S, **sc)
        assert_parity(got_o, got_l, ref_o, ref_l, f"fp8 bf16 q magnitudes {case} S={S}")
