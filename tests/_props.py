"""Properties every correct selection has, checked on the device at any size
(test-side only; nothing here is shared with the CUDA path or the oracle).

For a row (t, h) with v = min(M, num_valid_pages[t]) causal blocks and
n = min(K, v) slots in use ([47502] 实现拆解 and 关键源码片段; [55235]
执行摘要 for the total order):
  * slots [n, K) hold -1, slots [0, n) hold distinct ids in [0, v), ascending;
  * every init block [0, min(I, v)) and local block [max(v - L, 0), v) is
    selected;
  * exchange: no unselected causal block beats a selected non-forced one,
    where "beats" is a higher score in IEEE totalOrder, or an equal bit
    pattern and a lower id.
The total order is realised here by the signed integer key of the raw bits
with the magnitude bits of negative values flipped (IEEE 754-2019 5.10:
for same-sign values, ordering the bit patterns as sign-magnitude integers
is totalOrder).
"""
from __future__ import annotations

import torch


def order_keys(scores: torch.Tensor) -> torch.Tensor:
    """int32 keys whose signed order is totalOrder of the scores' bits."""
    if scores.dtype == torch.bfloat16:
        b = scores.view(torch.int16).to(torch.int32)
        return b ^ ((b >> 15) & 0x7FFF)
    b = scores.view(torch.int32)
    return b ^ ((b >> 31) & 0x7FFFFFFF)


def check_selection(scores: torch.Tensor, nvp: torch.Tensor, idx: torch.Tensor, K: int,
                    num_init: int, num_local: int, row_chunk: int = 1024) -> None:
    """Asserts the properties above for every row; scores [T, H, M] on the
    device, nvp int32 [T], idx int32 [T, H, K] (any strides)."""
    T, H, M = scores.shape
    dev = scores.device
    for t0 in range(0, T, row_chunk):
        t1 = min(T, t0 + row_chunk)
        sc = scores[t0:t1]
        ids = idx[t0:t1].to(torch.int64)
        v = torch.clamp(nvp[t0:t1].to(dev).to(torch.int64), min=0, max=M).view(-1, 1, 1)
        n = torch.clamp(v, max=K)
        slot = torch.arange(K, device=dev).view(1, 1, K)
        used = slot < n
        assert bool((ids[~used.expand_as(ids)] == -1).all()), "slots past n must hold -1"
        assert bool(((ids >= 0) & (ids < v) | ~used).all()), "ids must lie in [0, v)"
        asc = (ids[:, :, 1:] > ids[:, :, :-1]) | ~used[:, :, 1:]
        assert bool(asc.all()), "ids must be strictly ascending"
        # selected mask over the tiles (the -1 slots land in a spare column)
        sel = torch.zeros((t1 - t0, H, M + 1), dtype=torch.bool, device=dev)
        sel.scatter_(2, torch.where(used, ids, torch.full_like(ids, M)), True)
        sel = sel[:, :, :M]
        col = torch.arange(M, device=dev).view(1, 1, M)
        causal = col < v
        forced = causal & ((col < num_init) | (col >= v - num_local))
        assert not bool((forced & ~sel).any()), "an init or local block is missing"
        keys = order_keys(sc)
        big = torch.iinfo(torch.int32).max
        small = torch.iinfo(torch.int32).min
        chosen = sel & ~forced
        left = causal & ~sel
        kmin = torch.where(chosen, keys, torch.full_like(keys, big)).amin(dim=2)
        kmax = torch.where(left, keys, torch.full_like(keys, small)).amax(dim=2)
        assert bool((kmin >= kmax).all()), "an unselected block has a higher score"
        # equal keys at the boundary: every selected one has a lower id
        tie = (kmin == kmax).unsqueeze(2)
        at = keys == kmax.unsqueeze(2)
        hi_sel = torch.where(chosen & at & tie, col, torch.full_like(col, -1)).amax(dim=2)
        lo_left = torch.where(left & at & tie, col, torch.full_like(col, M)).amin(dim=2)
        assert bool((hi_sel < lo_left).all()), "a tie went to the higher block id"
