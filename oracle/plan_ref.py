"""Split-count heuristic, second statement (pure Python).  TEST INFRASTRUCTURE.

Source: "Flash-Decoding: Split-KV Attention for Long-Context Decode" (kanthi.in),
§6 "How many splits?", and the FlashAttention-3 comment quoted in the vatshank
split-KV post ("Benchmarking split-KV against vanilla FA" section): choose the
split count by wave efficiency -- how full the last wave of CTAs is -- and take
the smallest count within 85% of the best.

The arithmetic is Python's: true division of ints is correctly rounded, so each
efficiency is the IEEE double nearest the exact rational, the same value the C
statement (``fd_oracle.cpp``) and the library compute.
"""
from __future__ import annotations

import math


def efficiency_ref(work_items: int, slots: int, splits: int) -> float:
    """Busy fraction of the last wave when work_items*splits CTAs fill `slots`."""
    waves = work_items * splits / slots
    return waves / math.ceil(waves)


def num_splits_ref(work_items: int, slots: int, n_kv_blocks: int,
                   max_splits: int = 128) -> int:
    """Number of KV splits for `work_items` independent (batch, KV head) units."""
    if work_items >= 0.8 * slots:          # one pass already fills the machine
        return 1
    top = min(max_splits, slots, n_kv_blocks)
    candidates = {}
    for s in range(1, top + 1):
        # a count that gives the same blocks per split as s-1 buys nothing
        if s > 1 and math.ceil(n_kv_blocks / s) == math.ceil(n_kv_blocks / (s - 1)):
            continue
        candidates[s] = efficiency_ref(work_items, slots, s)
    if not candidates:                      # no KV blocks at all
        return 1
    best = max(candidates.values())
    return min(s for s, e in candidates.items() if e >= 0.85 * best)
