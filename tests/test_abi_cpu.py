"""The C-ABI library on the host: it loads, exports every symbol the header
declares, plans exactly like both statements of the heuristic in the oracle,
and rejects bad arguments before touching the GPU.  CPU only."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from plan_model import slot_model

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fd():
    import split_kv_gb300
    from split_kv_gb300 import _build
    _build.build()
    return split_kv_gb300


def _header_functions():
    src = open(os.path.join(ROOT, "include", "fd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(fd):
    declared = _header_functions()
    assert declared, "no functions parsed from include/fd.h"
    lib = ctypes.CDLL(fd.library_path())
    for name in declared:
        assert hasattr(lib, name), f"libfd.so does not export {name}"
    assert sorted(fd.EXPORTS) == declared


def test_abi_version_and_strings(fd):
    assert fd.fd_abi_version() == 4
    for code in range(-6, 1):
        s = fd.fd_status_string(code)
        assert s and s != "unknown status"
    assert fd.fd_status_string(99) == "unknown status"


def test_desc_struct_size_matches_header(fd):
    # 6 int32 + 9 int64 + 6 int32 + 1 int64 + 2 int32 + 2 float = 144 bytes
    assert ctypes.sizeof(fd.FdDesc) == 144
    assert fd.FdDesc.q_stride_t.offset == 120
    assert fd.FdDesc.k_scale.offset == 136 and fd.FdDesc.v_scale.offset == 140


def test_plan_splits_matches_oracle_table(fd, golden_dir):
    import json
    g = json.load(open(os.path.join(golden_dir, "fd_split_table_132sm.json")))
    for batch, heads, ctx, work, splits, _ in g["rows"]:
        assert fd.fd_plan_splits(work, g["slots"], -(-ctx // 128)) == splits
        assert fd.fd_plan(batch, heads, heads, 128, [ctx] * batch, 132) == splits


def test_plan_splits_equals_both_oracle_statements(fd):
    rng = np.random.default_rng(21)
    for slots in (264, 296, 304):
        for work in range(1, 260):
            for nb in (0, 1, 2, 5, 8, 31, 32, 33, 64, 100, 250, 256, 257, 1000, 1024, 2048, 2100):
                want = oracle.num_splits_ref(work, slots, nb)
                assert fd.fd_plan_splits(work, slots, nb) == want, (work, slots, nb)
    for _ in range(4000):
        w, s, nb, ms = (int(rng.integers(1, 600)), int(rng.integers(1, 500)),
                        int(rng.integers(0, 4000)), int(rng.integers(1, 200)))
        assert fd.fd_plan_splits(w, s, nb, ms) == oracle.plan(w, s, nb, ms)


def test_plan_for_the_workloads(fd):
    """Planned split counts of the five workloads at 148 and 152 SMs."""
    import fd_inputs
    W = fd_inputs.WORKLOADS
    for sms in (148, 152):
        slots = 2 * sms
        c = W["long_gqa_128k"]
        got = fd.fd_plan(1, 32, 8, 128, [c["ctx"]], sms)
        assert got == oracle.num_splits_ref(8, slots, -(-c["ctx"] // 128))
        L = fd_inputs.varlen_seqlens(W["varlen_b16"]["seed"])
        assert fd.fd_plan(16, 32, 8, 128, L, sms) == oracle.num_splits_ref(128, slots, -(-int(L.max()) // 128))
        assert fd.fd_plan(8, 64, 8, 128, [65536] * 8, sms) == oracle.num_splits_ref(64, slots, 512)
        for b in (1, 4, 16, 64):
            for ctx in (1024, 8192, 32768, 131072, 262144):
                assert fd.fd_plan(b, 32, 8, 128, [ctx] * b, sms) == \
                    oracle.num_splits_ref(8 * b, slots, -(-ctx // 128))
    assert fd.fd_plan(1, 32, 8, 128, [128000], 148) == 31
    assert fd.fd_plan(1, 32, 8, 128, [128000], 152) == 33


def test_plan_rejects_bad_arguments(fd):
    assert fd.fd_plan_splits(0, 264, 10) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan_splits(8, 0, 10) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan_splits(8, 264, -1) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan_splits(8, 264, 10, 0) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan(1, 32, 6, 128, [10], 148) == fd.FD_ERR_INVALID_ARG    # 6 does not divide 32
    assert fd.fd_plan(2, 32, 8, 128, [10, -1], 148) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan(1, 32, 8, 128, [0], 148) == 1                        # empty sequence


def test_plan_validates_an_optional_page_table(fd):
    """The decode contract plans from host lengths and, for a paged cache,
    the block table: a table never changes the plan, a table that misses a
    page or holds a negative page index where the sequence reaches is
    rejected."""
    sl = [100, 33, 0]
    bt = np.arange(3 * 8, dtype=np.int32).reshape(3, 8)
    want = fd.fd_plan(3, 32, 8, 128, sl, 148)
    assert want == oracle.num_splits_ref(24, 296, 1)
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=bt, page_size=16) == want
    for ps in (16, 64, 128):      # 100 tokens take 7, 2 and 1 of the 8 pages a row has
        assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=bt, page_size=ps) == want
    # 100 tokens need 13 pages of 8 but a row has 8
    small = np.zeros((3, 8), dtype=np.int32)
    assert fd.fd_plan(3, 32, 8, 128, [100, 1, 1], 148, block_table_host=small[:, :8],
                      page_size=8) == fd.FD_ERR_INVALID_ARG
    neg = bt.copy()
    neg[1, 2] = -1      # sequence 1 (33 tokens, 16-token pages) reaches page 2
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=neg, page_size=16) == fd.FD_ERR_INVALID_ARG
    neg = bt.copy()
    neg[1, 3] = -1      # ... but not page 3: unused entries are not read
    neg[2, 0] = -7      # and the empty sequence reads none
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=neg, page_size=16) == want
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=bt, page_size=12) == fd.FD_ERR_INVALID_ARG
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=bt, page_size=4) == fd.FD_ERR_UNSUPPORTED
    assert fd.fd_plan(3, 32, 8, 128, sl, 148, block_table_host=bt, page_size=0) == fd.FD_ERR_INVALID_ARG


def test_plan_desc_follows_the_slot_model_and_the_oracle(fd):
    """fd_plan_desc (the plan of fd_decode) against the oracle's statement of
    the heuristic fed the slot model above, over dtypes, flags, group sizes
    and query blocks; fd_plan is the same plan for a 16-bit cache, one query."""
    rng = np.random.default_rng(5)
    checked = 0
    for sms in (132, 148, 152):
        for G in (1, 2, 3, 4, 8, 16, 17, 24, 32, 64, 100, 128, 129, 256):
            for q_len in (1, 2, 4, 8, 16):
                if G * q_len > 256:
                    continue
                for fp8 in (False, True):
                    for cc in (False, True):
                        if cc and (fp8 or q_len != 1 or G not in (1, 2, 4, 8)):
                            continue
                        B = int(rng.integers(1, 20))
                        Hkv = int(rng.integers(1, 9))
                        L = rng.integers(0, 300000, size=B).astype(np.int32)
                        kw = dict(batch=B, n_q_heads=G * Hkv, n_kv_heads=Hkv, q_len=q_len,
                                  q_stride_t=G * Hkv * 128, q_stride_b=q_len * G * Hkv * 128,
                                  flags=fd.FD_FLAG_CUDA_CORES if cc else 0)
                        if fp8:
                            kw.update(kv_dtype=fd.FD_E4M3, q_dtype=fd.FD_F16, k_scale=1.0, v_scale=1.0)
                        d = _desc(fd, **kw)
                        work, slots = slot_model(B, Hkv, G, q_len, fp8, cc, sms)
                        want = oracle.num_splits_ref(work, slots, -(-int(L.max()) // 128))
                        assert fd.fd_plan_desc(d, L, sms) == want, (sms, G, q_len, fp8, cc, B, Hkv)
                        if q_len == 1 and not fp8 and not cc:
                            assert fd.fd_plan(B, G * Hkv, Hkv, 128, L, sms) == want
                        checked += 1
    assert checked > 300


def test_plan_of_wide_groups_matches_the_launch(fd):
    """A single query with 32 heads per KV head runs the tcgen05 CTA (one per
    SM): 16 sequences x 8 KV heads = 128 CTAs already cover 0.8 of 152 slots,
    so neither fd_plan nor fd_decode splits."""
    L = [131072] * 16
    assert fd.fd_plan(16, 256, 8, 128, L, 152) == 1
    d = _desc(fd, batch=16, n_q_heads=256, n_kv_heads=8, q_stride_b=256 * 128)
    assert fd.fd_plan_desc(d, L, 152) == 1
    # the same group over an fp8 cache: two column blocks per split, two slots per SM
    d8 = _desc(fd, batch=16, n_q_heads=256, n_kv_heads=8, q_stride_b=256 * 128,
               kv_dtype=fd.FD_E4M3, q_dtype=fd.FD_BF16, k_scale=1.0, v_scale=1.0)
    assert fd.fd_plan_desc(d8, L, 152) == oracle.num_splits_ref(16 * 8 * 2, 304, 1024)


def _desc(fd, **kw):
    d = fd.FdDesc()
    d.batch, d.n_q_heads, d.n_kv_heads, d.head_dim = 1, 32, 8, 128
    d.kv_dtype, d.out_dtype = fd.FD_F16, fd.FD_F32
    d.q_stride_b, d.q_stride_h = 32 * 128, 128
    d.k_stride_b, d.k_stride_h, d.k_stride_t = 8 * 1024 * 128, 1024 * 128, 128
    d.v_stride_b, d.v_stride_h, d.v_stride_t = 8 * 1024 * 128, 1024 * 128, 128
    d.kv_extent = 1024
    d.max_seqlen = 1024
    d.n_splits = 4
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_workspace_size_layout(fd):
    d = _desc(fd)
    rows, S, D = 32, 4, 128
    def r256(x):
        return (x + 255) // 256 * 256
    want = r256(rows * S * D * 4) + 2 * r256(rows * S * 4)
    assert fd.fd_workspace_size(d, 4) == want
    assert fd.fd_workspace_size(d, 129) == 0
    assert fd.fd_workspace_size(_desc(fd, head_dim=64), 4) == 0
    assert fd.fd_workspace_size(_desc(fd, n_kv_heads=5), 4) == 0


def test_workspace_size_for_query_blocks_and_fp8(fd):
    """rows = batch * q_len * n_q_heads for a query block; an fp8 cache
    changes nothing in the workspace (states are fp32 either way)."""
    def r256(x):
        return (x + 255) // 256 * 256
    for B, Hq, ql, S in ((1, 32, 4, 9), (3, 64, 8, 7), (2, 16, 16, 1)):
        d = _desc(fd, batch=B, n_q_heads=Hq, q_len=ql, q_stride_t=Hq * 128, q_stride_b=ql * Hq * 128)
        rows = B * ql * Hq
        want = r256(rows * S * 128 * 4) + 2 * r256(rows * S * 4)
        assert fd.fd_workspace_size(d, S) == want, (B, Hq, ql, S)
        d8 = _desc(fd, batch=B, n_q_heads=Hq, q_len=ql, q_stride_t=Hq * 128, q_stride_b=ql * Hq * 128,
                   kv_dtype=fd.FD_E4M3, q_dtype=fd.FD_BF16, k_scale=0.25, v_scale=4.0)
        assert fd.fd_workspace_size(d8, S) == want
    # a query block wider than the supported limits is invalid, so its size is 0
    assert fd.fd_workspace_size(_desc(fd, q_len=17, q_stride_t=32 * 128), 4) == 0


def test_decode_rejects_bad_arguments_without_a_gpu(fd):
    """Every rejection happens on the host, before any CUDA call."""
    fake = 1 << 20        # a 16-byte-aligned address that is never dereferenced
    ws = 1 << 21
    big = 1 << 30
    call = lambda d, **kw: fd.fd_decode(
        d, kw.get("q", fake), kw.get("k", fake), kw.get("v", fake), kw.get("sl", fake),
        kw.get("bt", None), kw.get("out", fake), kw.get("lse", fake), kw.get("ws", ws),
        kw.get("wsb", big), stream=0)
    assert call(None if False else _desc(fd, head_dim=64)) == fd.FD_ERR_UNSUPPORTED
    cc = fd.FD_FLAG_CUDA_CORES
    assert call(_desc(fd, n_q_heads=24, flags=cc)) == fd.FD_ERR_UNSUPPORTED  # G = 3 on CUDA cores
    assert call(_desc(fd, q_len=2, q_stride_t=32 * 128, flags=cc)) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, q_len=17, q_stride_t=32 * 128)) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, n_q_heads=8 * 40, q_len=8, q_stride_t=320 * 128)) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, q_len=-1)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, q_len=4, q_stride_t=100)) == fd.FD_ERR_INVALID_ARG
    e4 = dict(kv_dtype=fd.FD_E4M3, q_dtype=fd.FD_F16, k_scale=0.5, v_scale=2.0)
    assert call(_desc(fd, **dict(e4, q_dtype=fd.FD_E4M3))) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, **dict(e4, k_scale=float("inf")))) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, **e4, flags=cc)) == fd.FD_ERR_UNSUPPORTED          # fp8 on CUDA cores
    assert call(_desc(fd, **e4, k_stride_t=136)) == fd.FD_ERR_INVALID_ARG    # 136 B: not a 16 B multiple
    assert call(_desc(fd, reserved=1)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, n_q_heads=20)) == fd.FD_ERR_INVALID_ARG           # 8 does not divide 20
    assert call(_desc(fd, kv_dtype=fd.FD_F32)) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, kv_dtype=7)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, out_dtype=9)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, n_splits=129)) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, k_stride_t=100)) == fd.FD_ERR_INVALID_ARG          # not 16-byte multiple
    assert call(_desc(fd, flags=2)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, kv_extent=0)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, page_size=12, max_pages_per_seq=4)) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, page_size=4, max_pages_per_seq=4), bt=fake) == fd.FD_ERR_UNSUPPORTED
    assert call(_desc(fd, page_size=16, max_pages_per_seq=0), bt=fake) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd, page_size=16, max_pages_per_seq=64)) == fd.FD_ERR_INVALID_ARG   # no table
    assert call(_desc(fd), bt=fake) == fd.FD_ERR_INVALID_ARG                # table without paging
    assert call(_desc(fd), q=None) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd), k=fake + 8) == fd.FD_ERR_INVALID_ARG             # misaligned cache
    assert call(_desc(fd), out=None) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd), ws=None) == fd.FD_ERR_INVALID_ARG
    assert call(_desc(fd), ws=ws + 64) == fd.FD_ERR_WORKSPACE               # misaligned workspace
    assert call(_desc(fd), wsb=1024) == fd.FD_ERR_WORKSPACE                 # too small
    assert call(_desc(fd, batch=-1)) == fd.FD_ERR_INVALID_ARG
    # a zero-size batch is valid and enqueues nothing
    assert call(_desc(fd, batch=0)) == fd.FD_OK
    assert fd.fd_combine_states(_desc(fd, n_splits=0), ws, fake, fake, workspace_bytes=big,
                                stream=0) == fd.FD_ERR_INVALID_ARG
