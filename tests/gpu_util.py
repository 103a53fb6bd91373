"""Helpers for the GPU parity tests: run the C-ABI path with guard canaries
around every buffer it writes, and compare with the oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import split_kv_gb300 as fd
from plan_model import slot_model

GUARD = 256          # guard elements (or bytes) on each side of every written buffer
ATOL, RTOL = 2e-3, 1e-2
LSE_ATOL = 1e-3


class Guarded:
    """A device buffer with NaN / 0xA5 canaries on both sides."""

    def __init__(self, n: int, dtype, device, fill_float=float("nan"), align: int = 256):
        esz = torch.tensor([], dtype=dtype).element_size()
        pad = GUARD + align // esz
        self.full = torch.empty(n + 2 * pad, dtype=dtype, device=device)
        if dtype.is_floating_point:
            self.full.fill_(fill_float)
        else:
            self.full.fill_(0xA5)
        # first aligned element after the guard
        base = self.full.data_ptr()
        start = GUARD
        while (base + start * esz) % align:
            start += 1
        self.start, self.n = start, n
        self.view = self.full[start:start + n]
        self.before = self.full[:start].clone()
        self.after = self.full[start + n:].clone()

    def intact(self) -> bool:
        """Both canaries hold the exact bit patterns they were filled with."""
        def bits(t):
            esz = t.element_size()
            return t.view({4: torch.int32, 2: torch.int16, 1: torch.uint8}[esz])
        a = self.full[:self.start]
        b = self.full[self.start + self.n:]
        return torch.equal(bits(a), bits(self.before)) and torch.equal(bits(b), bits(self.after))


def run_decode(q, k, v, seqlens_h, *, n_kv_heads=None, page_size=0, block_table=None,
               n_splits=0, out_dtype=torch.float32, stream=None, check_guards=True, flags=0,
               k_scale=1.0, v_scale=1.0):
    """fd_decode through the C ABI; returns (out [rows, D] f64, lse [rows] f64, S)
    with rows = B*q_len*Hq (q is [B, Hq, D] or a query block [B, q_len, Hq, D])."""
    dev = q.device
    if q.dim() == 4:
        B, ql, Hq, D = q.shape
    else:
        (B, Hq, D), ql = q.shape, 1
    seqlens_h = np.asarray(seqlens_h, dtype=np.int32)
    seqlens = torch.from_numpy(seqlens_h).to(dev)
    bt = None
    mp = 0
    if page_size:
        bt = torch.from_numpy(np.ascontiguousarray(block_table, dtype=np.int32)).to(dev)
        mp = block_table.shape[1]
    desc = fd.make_desc(q, k, v, n_kv_heads=n_kv_heads, page_size=page_size, max_pages_per_seq=mp,
                        max_seqlen=int(seqlens_h.max()) if B else 0, n_splits=n_splits,
                        out_dtype=out_dtype, k_scale=k_scale, v_scale=v_scale)
    desc.flags = flags
    if n_splits > 0:
        S = n_splits
    else:
        # the planner's rule with the CTAs per split of this query block
        S = planned_splits(B, Hq, desc.n_kv_heads, ql, seqlens_h, fp8=desc.kv_dtype == fd.FD_E4M3,
                           cuda_cores=(flags & fd.FD_FLAG_CUDA_CORES) != 0)
        if B > 0:
            assert S == fd.fd_plan_desc(desc, seqlens_h)
        if B > 0 and ql == 1 and desc.kv_dtype != fd.FD_E4M3 and not flags & fd.FD_FLAG_CUDA_CORES:
            assert S == fd.fd_plan(B, Hq, desc.n_kv_heads, D, seqlens_h)
    assert S >= 1
    desc.n_splits = 0 if n_splits <= 0 else S
    wsb = fd.fd_workspace_size(desc, 0)
    assert wsb == fd.fd_workspace_size(desc, S) > 0
    out = Guarded(B * ql * Hq * D, out_dtype, dev)
    lse = Guarded(B * ql * Hq, torch.float32, dev)
    ws = Guarded(wsb, torch.uint8, dev)
    fd.check(fd.fd_decode(desc, q, k, v, seqlens, bt, out.view, lse.view, ws.view, wsb,
                          stream=stream), "fd_decode")
    fd.check(fd.fd_device_status(stream), "device status")
    torch.cuda.synchronize()
    if check_guards:
        assert out.intact(), "fd_decode wrote outside out"
        assert lse.intact(), "fd_decode wrote outside lse"
        assert ws.intact(), "fd_decode wrote outside its workspace"
    o = out.view.float().cpu().double().numpy().reshape(B * ql * Hq, D)
    l = lse.view.cpu().double().numpy()
    return o, l, S


def planned_splits(B, Hq, Hkv, q_len, seqlens_h, fp8=False, cuda_cores=False):
    """n_splits fd_decode should plan: the oracle's statement of the heuristic
    fed the launch shape of plan_model (this GPU's SM count)."""
    work, slots = slot_model(B, Hkv, Hq // Hkv, q_len, fp8, cuda_cores, fd.fd_num_sms())
    blocks = -(-int(np.max(seqlens_h)) // 128) if B else 0
    return oracle.num_splits_ref(work, slots, blocks)


def assert_parity(got_o, got_l, ref_o, ref_l, what=""):
    assert not np.isnan(got_o).any(), f"{what}: NaN in out"
    assert not np.isnan(got_l).any(), f"{what}: NaN in lse"
    err = np.abs(got_o - ref_o)
    tol = ATOL + RTOL * np.abs(ref_o)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance, max abs err "
                           f"{err.max():.3e}")
    fin = np.isfinite(ref_l)
    assert np.all(np.isneginf(got_l[~fin])), f"{what}: lse of empty rows must be -inf"
    assert np.all(np.isfinite(got_l[fin])), f"{what}: non-finite lse"
    if fin.any():
        le = np.abs(got_l[fin] - ref_l[fin]).max()
        assert le <= LSE_ATOL, f"{what}: lse err {le:.3e}"
    return float(err.max()) if err.size else 0.0


def oracle_all(q, k, v, seqlens_h, dtype, n_kv_heads, page_size=0, block_table=None, rows=None,
               kv_dtype=None, k_scale=1.0, v_scale=1.0):
    return oracle.decode(q.cpu(), k.cpu(), v.cpu(), seqlens_h, dtype=dtype, n_kv_heads=n_kv_heads,
                         page_size=page_size, block_table=block_table, rows=rows,
                         kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale)


def oracle_rows_contiguous(q, k, v, seqlens_h, rows, dtype):
    """Oracle on selected rows of a huge contiguous cache: copies each
    (b, kv head) slice the rows read once."""
    B, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = [int(r) for r in rows]
    res = {}
    groups = {}
    for r in rows:
        b, h = divmod(r, Hq)
        groups.setdefault((b, h // G), []).append(h)
    for (b, g), heads in groups.items():
        L = int(seqlens_h[b])
        kk = k[b:b + 1, g:g + 1, :max(L, 1)].cpu()
        vv = v[b:b + 1, g:g + 1, :max(L, 1)].cpu()
        qq = q[b:b + 1, heads].cpu()
        o, l = oracle.decode(qq, kk, vv, [L], dtype=dtype, n_kv_heads=1)
        for i, h in enumerate(heads):
            res[b * Hq + h] = (o[i], l[i])
    return np.stack([res[r][0] for r in rows]), np.array([res[r][1] for r in rows])
