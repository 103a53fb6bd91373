"""Seeded synthetic inputs for split-KV decode attention.

This module is shared by the tests, the smoke check and the bench.  It holds
only shapes, seeds and random draws -- none of the method's arithmetic -- so
that the oracle and the CUDA path can be fed the same bytes without sharing
any code.

Workloads (the pages measure on no dataset; every input is synthetic):
  tiny_mha       B=1, 8 q heads = 8 KV heads, d=128, context 4096, fp16.
  long_gqa_128k  B=1, 32 q heads over 8 KV heads, d=128, context 128000, fp16,
                 32 layers with distinct caches (the headline workload:
                 "Flash-Decoding: Split-KV Attention for Long-Context Decode",
                 §1 worked numbers, 524 MB of K+V per layer).
  varlen_b16     B=16, 32 / 8 heads, d=128, bf16, lengths uniform in
                 [1, 32768] with forced ragged cases.
  paged_b8       B=8, 64 / 8 heads, d=128, bf16, 65536 tokens each, pages of
                 16 tokens, block table a seeded permutation of a shared pool.
  sweep          batch {1,4,16,64} x context {1K,8K,32K,128K,256K}, 32 / 8
                 heads, d=128, fp16.
  query_block_q4 B=4, 32 / 8 heads, d=128, bf16, 32768 tokens, 4 query
                 positions per sequence (a speculative-verification block).
  query_block_g8_q4, query_block_g8_q8, query_block_g16_q8  the same cache
                 with 64 or 128 query heads and 4 or 8 positions: 32, 64 and
                 128 (position, head) columns per KV head.
  long_gqa_128k_fp8  the headline shape with an E4M3 cache (q fp16), values
                 stored x64 with k_scale = v_scale = 1/64.
  sweep_fp8     the sweep's grid over such an E4M3 cache.
K, V and q are i.i.d. N(0,1) cast to the cache dtype.
"""
from __future__ import annotations

import numpy as np

TILE_TOKENS = 128  # not used for arithmetic: only to force lengths at tile edges

WORKLOADS = {
    "tiny_mha": dict(batch=1, n_q_heads=8, n_kv_heads=8, head_dim=128, ctx=4096,
                     dtype="f16", seed=1001, forced_splits=(1, 3, 7)),
    "long_gqa_128k": dict(batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, ctx=128000,
                          dtype="f16", seed=1002, layers=32),
    "varlen_b16": dict(batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, ctx=32768,
                       dtype="bf16", seed=1003),
    "paged_b8": dict(batch=8, n_q_heads=64, n_kv_heads=8, head_dim=128, ctx=65536,
                     dtype="bf16", seed=1004, page_size=16),
    "sweep": dict(batches=(1, 4, 16, 64), ctxs=(1024, 8192, 32768, 131072, 262144),
                  n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="f16", seed=1005),
    # the same grid over an E4M3 cache (q fp16), values stored x64, scales 1/64
    "sweep_fp8": dict(batches=(1, 4, 16, 64), ctxs=(1024, 8192, 32768, 131072, 262144),
                      n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="f16", kv_dtype="e4m3",
                      kv_gain=64.0, seed=1008),
    # the headline shape with an fp8 (E4M3) cache, one scale per tensor:
    # stored = value * kv_gain, k_scale = v_scale = 1 / kv_gain
    "long_gqa_128k_fp8": dict(batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, ctx=128000,
                              dtype="f16", kv_dtype="e4m3", kv_gain=64.0, seed=1007, layers=32),
    # short query block (speculative verification of 4 draft tokens)
    "query_block_q4": dict(batch=4, n_q_heads=32, n_kv_heads=8, head_dim=128, ctx=32768,
                           q_len=4, dtype="bf16", seed=1006),
    # wider blocks: a group of 8 query heads per KV head, 4 or 8 positions
    # (32 and 64 columns per KV head), and 16 heads x 8 positions (128 columns)
    "query_block_g8_q4": dict(batch=4, n_q_heads=64, n_kv_heads=8, head_dim=128, ctx=32768,
                              q_len=4, dtype="bf16", seed=1009),
    "query_block_g8_q8": dict(batch=4, n_q_heads=64, n_kv_heads=8, head_dim=128, ctx=32768,
                              q_len=8, dtype="bf16", seed=1010),
    "query_block_g16_q8": dict(batch=4, n_q_heads=128, n_kv_heads=8, head_dim=128, ctx=32768,
                               q_len=8, dtype="bf16", seed=1011),
}


def torch_dtype(name: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


def randn(shape, dtype: str, seed: int, device="cpu", gain: float = 1.0):
    """N(0, gain^2) draws cast to fp16 / bf16, from a seeded torch generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if gain != 1.0:
        x.mul_(gain)
    return x.to(torch_dtype(dtype))


def varlen_seqlens(seed: int, batch: int = 16, max_len: int = 32768) -> np.ndarray:
    """Lengths uniform in [1, max_len], then forced ragged cases: a length-1
    sequence, one tile minus / plus one, a full-capacity sequence and k*tile+1."""
    rng = np.random.default_rng(seed)
    L = rng.integers(1, max_len + 1, size=batch).astype(np.int32)
    forced = [1, TILE_TOKENS - 1, TILE_TOKENS + 1, max_len, TILE_TOKENS * 37 + 1]
    for i, v in enumerate(forced[:batch]):
        L[i] = min(v, max_len)
    return L


def page_permutation(seed: int, n_pages: int) -> np.ndarray:
    """A seeded random permutation of physical page ids 0..n_pages-1."""
    rng = np.random.default_rng(seed)
    return rng.permutation(n_pages).astype(np.int32)


def block_table(seed: int, batch: int, pages_per_seq: int, n_pages: int | None = None):
    """block_table[b][j] = perm[b * pages_per_seq + j] over a pool of n_pages pages."""
    n_pages = n_pages or batch * pages_per_seq
    perm = page_permutation(seed, n_pages)
    return perm[: batch * pages_per_seq].reshape(batch, pages_per_seq).copy()


def randn_chunked(shape, dtype: str, seed: int, device="cpu", gain: float = 1.0):
    """Like randn, but drawn one leading index at a time (seed*1000003 + i), so
    caches of tens of GB need only one slice of f32 scratch."""
    import torch
    out = torch.empty(*shape, dtype=torch_dtype(dtype), device=device)
    g = torch.Generator(device=device)
    for i in range(shape[0]):
        g.manual_seed(int(seed) * 1000003 + i)
        x = torch.randn(*shape[1:], generator=g, device=device, dtype=torch.float32)
        if gain != 1.0:
            x.mul_(gain)
        out[i].copy_(x)
        del x
    return out


def randn_fp8(shape, seed: int, device="cpu", gain: float = 1.0):
    """N(0, gain^2) draws clamped to the E4M3 range (+-448) and stored as
    torch.float8_e4m3fn, drawn one leading index at a time like randn_chunked."""
    import torch
    out = torch.empty(*shape, dtype=torch.float8_e4m3fn, device=device)
    g = torch.Generator(device=device)
    for i in range(shape[0]):
        g.manual_seed(int(seed) * 1000003 + i)
        x = torch.randn(*shape[1:], generator=g, device=device, dtype=torch.float32)
        x.mul_(gain).clamp_(-448.0, 448.0)
        out[i].copy_(x)
        del x
    return out
