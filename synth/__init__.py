"""Seeded synthetic inputs for the top-k selection path.

This module is shared by the tests (oracle side and CUDA side) and the
benchmark.  It draws random numbers and lays out buffers; it holds none of
the method's arithmetic: no causal page count, no row-to-request mapping, no
ordering of scores.  Where an input depends on the causal page count (the
-inf tail of unwritten tiles, a block planted at a causal position), the
caller computes the count on its own side and passes it in.

The shapes and value distributions follow the workloads of the vLLM MiniMax-M3
PR reports: the production 8k+1k decode graph with a 74-block capacity,
decode query lengths 1-4, 1-4 index heads, topk 16, long contexts up to 1024
blocks, a mixed decode+prefill unified buffer, and the speculative-decode
sparse block table.  Nothing here stands in for a public dataset: the pages
measure on none.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

# IEEE bit patterns injected as special scores.
BF16_SPECIALS = {
    "+nan": 0x7FC0, "-nan": 0xFFC0, "+nan_payload": 0x7F81, "-nan_payload": 0xFF81,
    "+inf": 0x7F80, "-inf": 0xFF80, "+0": 0x0000, "-0": 0x8000,
}
FP32_SPECIALS = {
    "+nan": 0x7FC00000, "-nan": 0xFFC00000, "+nan_payload": 0x7F800001,
    "-nan_payload": 0xFF800001, "+inf": 0x7F800000, "-inf": 0xFF800000,
    "+0": 0x00000000, "-0": 0x80000000,
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_scores(shape, dtype: torch.dtype, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) scores drawn in fp32 and rounded (nearest-even) to `dtype`."""
    g = generator(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def _bits_view(scores: torch.Tensor) -> torch.Tensor:
    if scores.dtype == torch.bfloat16:
        return scores.view(torch.int16)
    if scores.dtype == torch.float32:
        return scores.view(torch.int32)
    raise TypeError(scores.dtype)


def _as_signed(bits: int, width: int) -> int:
    return bits - (1 << width) if bits >= (1 << (width - 1)) else bits


def inject_specials(scores: torch.Tensor, seed: int, frac_each: float = 0.01,
                    frac_ties: float = 0.01) -> torch.Tensor:
    """In place: set about `frac_each` of the elements to each special bit
    pattern (NaNs with and without payload, +-Inf, +-0) and copy the bits of
    the left neighbour into about `frac_ties` of them (exact ties)."""
    g = generator(seed, scores.device)
    bits = _bits_view(scores)
    table = BF16_SPECIALS if scores.dtype == torch.bfloat16 else FP32_SPECIALS
    width = 16 if scores.dtype == torch.bfloat16 else 32
    u = torch.rand(scores.shape, generator=g, device=scores.device)
    lo = 0.0
    for pattern in table.values():
        sel = (u >= lo) & (u < lo + frac_each)
        bits[sel] = _as_signed(pattern, width)
        lo += frac_each
    tie = torch.rand(scores.shape, generator=g, device=scores.device) < frac_ties
    tie[..., 0] = False
    left = torch.roll(bits, shifts=1, dims=-1)
    bits[tie] = left[tie]
    return scores


def fill_tail(scores: torch.Tensor, counts: torch.Tensor, value: float) -> torch.Tensor:
    """In place: scores[t, h, b] = value for b >= counts[t] (the caller's
    per-token count of written tiles)."""
    M = scores.shape[-1]
    cols = torch.arange(M, device=scores.device).view(1, 1, M)
    mask = cols >= counts.to(scores.device).view(-1, 1, 1).long()
    scores.masked_fill_(mask.expand_as(scores), value)
    return scores


def plant(scores: torch.Tensor, counts: torch.Tensor, u: torch.Tensor, value: float) -> torch.Tensor:
    """In place: for each row (t, h) with counts[t] > 0 write `value` at
    column floor(u[t, h] * counts[t])."""
    T, H, M = scores.shape
    c = counts.to(scores.device).long().view(T, 1).expand(T, H)
    col = torch.clamp((u.to(scores.device) * c).floor().long(), max=M - 1)
    ok = c > 0
    t_idx = torch.arange(T, device=scores.device).view(T, 1).expand(T, H)
    h_idx = torch.arange(H, device=scores.device).view(1, H).expand(T, H)
    scores[t_idx[ok], h_idx[ok], col[ok]] = torch.tensor(value, dtype=scores.dtype,
                                                         device=scores.device)
    return scores


@dataclass
class Workload:
    """One synthetic workload.  Decode workloads carry `seq_lens` (+ `dql`);
    varlen workloads carry `cu_seqlens_q` and `prefix_lens` instead."""
    name: str
    dtype: torch.dtype
    T: int
    H: int
    M: int
    K: int
    num_init: int
    num_local: int
    scores: torch.Tensor                      # [T, H, M], every tile drawn
    dql: int = 1
    seq_lens: torch.Tensor | None = None      # int32 [B]
    cu_seqlens_q: torch.Tensor | None = None  # int32 [N+1]
    prefix_lens: torch.Tensor | None = None   # int32 [N]
    block_table: torch.Tensor | None = None   # int32 [B, MB]
    plant_u: torch.Tensor | None = None       # float [T, H] in [0, 1)
    plant_value: float | None = None
    notes: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return 0 if self.seq_lens is None else int(self.seq_lens.shape[0])


def _uniform_int(lo: int, hi: int, n: int, g: torch.Generator, device) -> torch.Tensor:
    """n integers uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (n,), generator=g, device=device, dtype=torch.int64)


def tiny_decode(seed: int = 1001, device="cpu") -> Workload:
    """8 requests, decode query length 1, one index head, 16-tile capacity,
    topk 4, fp32 N(0,1), seq_len uniform in [1, 2048]."""
    g = generator(seed, device)
    seq = _uniform_int(1, 2048, 8, g, device).to(torch.int32)
    sc = normal_scores((8, 1, 16), torch.float32, seed + 17, device)
    return Workload("tiny_decode", torch.float32, 8, 1, 16, 4, 1, 1, sc, dql=1, seq_lens=seq)


def short_decode(seed: int = 1002, device="cpu", B: int = 64, dql: int = 4, H: int = 4,
                 M: int = 74, K: int = 16, dtype=torch.bfloat16) -> Workload:
    """Production short-context decode: 64 requests x query length 4, 4 index
    heads, 74-tile capacity (8k+1k context), topk 16, bf16 N(0,1) with about
    1% of each special value and 1% exact ties, about 5% padded requests
    (seq_len 0), about a quarter of the requests placed so that their query
    rows straddle a multiple of 128, and a few shorter than the query length."""
    g = generator(seed, device)
    cap = M * 128
    seq = _uniform_int(dql + 1, cap, B, g, device)
    kind = torch.rand(B, generator=g, device=device)
    m = _uniform_int(1, M - 1, B, g, device)
    off = _uniform_int(1, dql, B, g, device)
    straddle = (kind < 0.25)
    seq = torch.where(straddle, m * 128 + off, seq)
    short = (kind >= 0.25) & (kind < 0.30)
    seq = torch.where(short, _uniform_int(1, max(1, dql - 1), B, g, device), seq)
    padded = (kind >= 0.30) & (kind < 0.35)
    seq = torch.where(padded, torch.zeros_like(seq), seq)
    seq = seq.clamp(max=cap).to(torch.int32)
    sc = normal_scores((B * dql, H, M), dtype, seed + 17, device)
    inject_specials(sc, seed + 29)
    return Workload("short_decode", dtype, B * dql, H, M, K, 1, 1, sc, dql=dql, seq_lens=seq)


def long_decode(seed: int = 1003, device="cpu", B: int = 128, H: int = 2, M: int = 1024,
                K: int = 16, dtype=torch.bfloat16, min_len: int = 16384,
                max_len: int = 131072, num_local: int = 2) -> Workload:
    """Long-context decode: query length 1, seq_len uniform in
    [16384, 131072] (up to 1024 blocks), bf16 N(0,1) plus one planted block
    (+8.0) per row at a uniform causal position; 1 init and 2 local blocks."""
    g = generator(seed, device)
    seq = _uniform_int(min_len, max_len, B, g, device).to(torch.int32)
    sc = normal_scores((B, H, M), dtype, seed + 17, device)
    u = torch.rand((B, H), generator=g, device=device)
    return Workload("long_decode", dtype, B, H, M, K, 1, num_local, sc, dql=1, seq_lens=seq,
                    plant_u=u, plant_value=8.0)


def mixed_prefill_decode(seed: int = 1004, device="cpu", num_decode: int = 32,
                         prefill_lens=(8192, 8192), H: int = 4, M: int = 128, K: int = 16,
                         dtype=torch.float32, prefill_prefix=None,
                         decode_max_prefix: int = 16383) -> Workload:
    """Unified buffer: 32 decode tokens (one per request, context before the
    token uniform in [0, 16383]) followed by two 8192-token prefills from
    position 0; 4 index heads, 128-tile capacity, topk 16, fp32 N(0,1).
    `prefill_prefix` gives each prefill chunk the context that precedes it
    (default none), and `decode_max_prefix` the largest decode context, so
    the same layout also describes long-context batches at a large capacity."""
    g = generator(seed, device)
    dec_prefix = _uniform_int(0, decode_max_prefix, num_decode, g, device)
    qlens = [1] * num_decode + list(prefill_lens)
    cu = torch.tensor([0] + list(torch.tensor(qlens).cumsum(0).tolist()), dtype=torch.int32,
                      device=device)
    pre = [0] * len(prefill_lens) if prefill_prefix is None else list(prefill_prefix)
    prefix = torch.cat([dec_prefix, torch.tensor(pre, dtype=torch.int64,
                                                 device=device)]).to(torch.int32)
    T = int(cu[-1])
    sc = normal_scores((T, H, M), dtype, seed + 17, device)
    return Workload("mixed_prefill_decode", dtype, T, H, M, K, 1, 1, sc, cu_seqlens_q=cu,
                    prefix_lens=prefix, notes={"num_decode": num_decode})


def fused_table(seed: int = 1005, device="cpu", B: int = 256, dql: int = 4, H: int = 1,
                M: int = 512, K: int = 16, dtype=torch.bfloat16, max_len: int = 65536,
                distinct_blocks: bool = True) -> Workload:
    """Fused select + sparse block table: 256 requests x query length 4, one
    index head, seq_len uniform in [1, 65536] with about 5% padded (0),
    block_table [256, 512] of distinct physical block ids (a seeded
    permutation of [0, 131072)), topk 16."""
    g = generator(seed, device)
    seq = _uniform_int(1, max_len, B, g, device)
    padded = torch.rand(B, generator=g, device=device) < 0.05
    seq = torch.where(padded, torch.zeros_like(seq), seq).to(torch.int32)
    if distinct_blocks:
        perm = torch.randperm(B * M, generator=g, device=device)
        bt = perm.view(B, M).to(torch.int32)
    else:
        bt = torch.randint(0, 1 << 27, (B, M), generator=g, device=device, dtype=torch.int32)
    sc = normal_scores((B * dql, H, M), dtype, seed + 17, device)
    return Workload("fused_table", dtype, B * dql, H, M, K, 1, 1, sc, dql=dql, seq_lens=seq,
                    block_table=bt)


def random_block_table(B: int, MB: int, seed: int, device="cpu") -> torch.Tensor:
    """Physical block ids drawn uniformly from [0, 2^27) (so id*8+7 fits int32)."""
    g = generator(seed, device)
    return torch.randint(0, 1 << 27, (B, MB), generator=g, device=device, dtype=torch.int32)


def index_inputs(seed: int, T: int, H: int, D: int, num_phys_blocks: int, device="cpu",
                 integer_valued: bool = False):
    """Index queries bf16 [T, H, D] drawn N(0, 1/D) and pooled index keys bf16
    [num_phys_blocks, D] drawn N(0, 1), so that a block score (a dot product
    over D) is about N(0, 1) like the score workloads above.  With
    `integer_valued`, both hold integers in [-3, 3] instead: every product
    and partial sum is then an integer below 2^24, exact in fp32 whatever
    the summation order, and equal scores (ties) are common."""
    g = generator(seed, device)
    if integer_valued:
        q = torch.randint(-3, 4, (T, H, D), generator=g, device=device).float()
        k = torch.randint(-3, 4, (num_phys_blocks, D), generator=g, device=device).float()
    else:
        q = torch.randn(T, H, D, generator=g, device=device) / (D ** 0.5)
        k = torch.randn(num_phys_blocks, D, generator=g, device=device)
    return q.to(torch.bfloat16), k.to(torch.bfloat16)


def paged_block_table(B: int, MB: int, num_phys_blocks: int, seed: int, frac_missing: float = 0.0,
                      device="cpu") -> torch.Tensor:
    """int32 [B, MB] of distinct physical block ids from [0, num_phys_blocks)
    (a seeded permutation), with about `frac_missing` of the entries set to
    -1 or to an id past the end."""
    g = generator(seed, device)
    perm = torch.randperm(num_phys_blocks, generator=g, device=device)[:B * MB]
    bt = perm.view(B, MB).to(torch.int32)
    if frac_missing > 0:
        u = torch.rand((B, MB), generator=g, device=device)
        bt = torch.where(u < frac_missing / 2, torch.full_like(bt, -1), bt)
        bt = torch.where((u >= frac_missing / 2) & (u < frac_missing),
                         torch.full_like(bt, num_phys_blocks + 5), bt)
    return bt
