"""Pin checks for the CPU oracle: each check compares the oracle with
something other than itself (a value the pages print, a clause of IEEE 754,
a closed form, brute force on tiny inputs, a library sort on a special case).

Every check takes the ctypes library to test, so that the mutant test can run
the same checks against copies of the oracle with planted mistakes.
"""
from __future__ import annotations

import json
import os
import random

import numpy as np

import oracle
from tests import _pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_bits(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                out.append(int(line, 16))
    return out


def check_total_order_golden(lib=None):
    """IEEE 754-2019 5.10 order of hand-listed bit patterns (bf16 and fp32)."""
    for name, dtype in (("total_order_bf16.txt", oracle.BF16), ("total_order_fp32.txt", oracle.FP32)):
        seq = _read_bits(name)
        for i, a in enumerate(seq):
            for j, b in enumerate(seq):
                want = (i > j) - (i < j)
                got = oracle.total_order_cmp(a, b, dtype, lib=lib)
                assert got == want, f"{name}: cmp({a:#x}, {b:#x}) = {got}, want {want}"


def check_total_order_exhaustive_bf16(lib=None):
    """Every bf16 bit pattern, sorted by an independent Python key (float
    widening by bit shift); the oracle must agree on each adjacent pair."""
    pats = sorted(range(1 << 16), key=lambda b: _pins.order_key(b, True))
    keys = [_pins.order_key(b, True) for b in pats]
    for a, b, ka, kb in zip(pats, pats[1:], keys, keys[1:]):
        want = -1 if ka < kb else 0
        got = oracle.total_order_cmp(a, b, oracle.BF16, lib=lib)
        assert got == want, f"cmp({a:#06x}, {b:#06x}) = {got}, want {want}"


def check_total_order_random_fp32(lib=None, n=20000, seed=5):
    rng = random.Random(seed)
    specials = _read_bits("total_order_fp32.txt")
    for _ in range(n):
        a = rng.choice(specials) if rng.random() < 0.2 else rng.getrandbits(32)
        b = rng.choice(specials) if rng.random() < 0.2 else rng.getrandbits(32)
        ka, kb = _pins.order_key(a, False), _pins.order_key(b, False)
        want = (ka > kb) - (ka < kb)
        got = oracle.total_order_cmp(a, b, oracle.FP32, lib=lib)
        assert got == want, f"cmp({a:#x}, {b:#x}) = {got}, want {want}"


def check_causal_pages_golden(lib=None):
    rows = []
    with open(os.path.join(GOLDEN, "causal_pages.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                p, n = line.split()
                rows.append((int(p), int(n)))
    # decode form, query length 1: position = seq_len - 1
    for pos, pages in rows:
        got = oracle.num_valid_pages_decode([pos + 1], 1, lib=lib)[0]
        assert got == pages, f"decode pos {pos}: {got} != {pages}"
    # decode form, query length 8: the row of local_q = 7 sits at seq_len - 1
    for pos, pages in rows:
        got = oracle.num_valid_pages_decode([pos + 1], 8, lib=lib)[7]
        assert got == pages, f"decode dql=8 pos {pos}: {got} != {pages}"
    # varlen form: one-token sequences at position prefix_len
    ok = [(p, n) for p, n in rows if p >= 0]
    cu = list(range(len(ok) + 1))
    got = oracle.num_valid_pages_varlen(cu, [p for p, _ in ok], lib=lib)
    assert list(got) == [n for _, n in ok], (list(got), ok)


def check_varlen_prefill_positions(lib=None):
    """A 300-token chunk after a 100-token prefix: positions 100..399."""
    got = oracle.num_valid_pages_varlen([0, 300], [100], lib=lib)
    want = [(100 + j + 1 + 127) // 128 for j in range(300)]  # closed form of ceil
    assert list(got) == want


def _worked_example():
    with open(os.path.join(GOLDEN, "spec_decode_sparse_table.json")) as f:
        return json.load(f)


def check_spec_decode_worked_example(lib=None):
    ex = _worked_example()
    dql = ex["decode_query_len"]
    idx = np.array(ex["topk_idx"], dtype=np.int32)[:, None, :]
    bt, ctx = oracle.build_sparse_block_table(idx, ex["block_table"], ex["seq_lens"], dql, lib=lib)
    assert list(ctx[:, 0]) == ex["expected_ctx"], list(ctx[:, 0])
    width = ex["row_width"]
    assert bt.shape == (12, 1, width)
    for r, pref in enumerate(ex["expected_bt_nonzero_prefix"]):
        want = pref + [0] * (width - len(pref))
        assert list(bt[r, 0]) == want, (r, list(bt[r, 0]))
    # the page's padded-request rows: empty context, all-zero table
    assert (bt[8:] == 0).all() and (ctx[8:] == 0).all()
    nvp = oracle.num_valid_pages_decode(ex["seq_lens"], dql, lib=lib)
    assert list(nvp) == [3, 3, 3, 3, 2, 2, 2, 2, 0, 0, 0, 0]


def check_table_duplicates_ignored(lib=None):
    """A repeated id counts once (same table and ctx as the deduplicated row)."""
    seq = [700]
    table = [[3, 9, 27, 81, 243, 729]]
    a = np.array([[[4, 1, 4, 1, 5, -1]]], dtype=np.int32)
    b = np.array([[[4, 1, 5, -1, -1, -1]]], dtype=np.int32)
    ta, ca = oracle.build_sparse_block_table(a, table, seq, 1, lib=lib)
    tb, cb = oracle.build_sparse_block_table(b, table, seq, 1, lib=lib)
    assert (ta == tb).all() and (ca == cb).all()
    # position 699, causal 700: blocks 1, 4 full (256), block 5 holds 60 tokens
    assert ca[0, 0] == 128 + 128 + 60
    row = list(ta[0, 0])
    assert row[:8] == [9 * 8 + p for p in range(8)]
    assert row[8:16] == [243 * 8 + p for p in range(8)]
    assert row[16:20] == [729 * 8 + p for p in range(4)] and row[20:24] == [0] * 4


def check_table_full_selection_covers_causal_len(lib=None, seed=3):
    """When every causal block is selected, ctx equals the causal length and
    the table is the request's block list expanded page by page."""
    rng = np.random.default_rng(seed)
    for _ in range(50):
        dql = int(rng.integers(1, 5))
        seq = int(rng.integers(0, 2000))
        nblk = 20
        table = rng.integers(0, 1 << 20, size=(1, nblk)).astype(np.int32)
        K = nblk
        ids = np.tile(np.arange(K, dtype=np.int32), (dql, 1))[:, None, :]
        bt, ctx = oracle.build_sparse_block_table(ids, table, [seq], dql, lib=lib)
        for q in range(dql):
            causal = max(seq - dql + q + 1, 0)
            assert ctx[q, 0] == causal
            npages = -(-causal // 16)
            flat = [int(table[0, p // 8]) * 8 + p % 8 for p in range(npages)]
            assert list(bt[q, 0, :npages]) == flat
            assert (bt[q, 0, npages:] == 0).all()


def check_table_input_order_irrelevant(lib=None, seed=21):
    """The table keeps the valid distinct ids in ascending order ([47984]
    sections 实现拆解 item 3 and 关键源码片段, under the ascending reading), so
    reordering a row's ids changes nothing; a row of one repeated id gives
    the table of that id alone; and each kept block's entries come in
    ascending block order."""
    rng = np.random.default_rng(seed)
    for _ in range(40):
        K = int(rng.integers(2, 65))
        nblk = 96
        seq = int(rng.integers(0, nblk * 128 + 100))
        table = rng.permutation(1 << 20)[:nblk].astype(np.int32)[None, :]  # distinct
        row = rng.integers(-2, nblk + 3, size=K).astype(np.int32)
        rows = [row, row[::-1].copy(), rng.permutation(row)]
        outs = [oracle.build_sparse_block_table(r[None, None, :], table, [seq], 1, lib=lib)
                for r in rows]
        for bt, ctx in outs[1:]:
            assert (bt == outs[0][0]).all() and (ctx == outs[0][1]).all()
        bt = outs[0][0][0, 0]
        block_of = {int(table[0, b]) * 8: b for b in range(nblk)}
        kept = sorted({int(x) for x in row if 0 <= x < min(-(-seq // 128), nblk)})
        assert [block_of.get(int(bt[8 * j]), -1) for j in range(len(kept))] == kept
        b = int(rng.integers(0, nblk))
        same = np.full((1, 1, K), b, dtype=np.int32)
        one = np.full((1, 1, K), -1, dtype=np.int32)
        one[0, 0, 0] = b
        t1, c1 = oracle.build_sparse_block_table(same, table, [seq], 1, lib=lib)
        t2, c2 = oracle.build_sparse_block_table(one, table, [seq], 1, lib=lib)
        assert (t1 == t2).all() and (c1 == c2).all()


def _rand_row_bits(rng, v, is_bf16, palette_frac=0.5):
    """Row of bit patterns mixing a small palette (ties, NaN, +-0, +-Inf) and
    random finite values."""
    if is_bf16:
        pal = [0x7FC0, 0xFFC0, 0x7F81, 0xFF81, 0x7F80, 0xFF80, 0x0000, 0x8000, 0x3F80,
               0xBF80, 0x4000, 0x3F80]
        rnd = lambda: int(rng.integers(0, 1 << 16))
    else:
        pal = [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7F800000, 0xFF800000,
               0x0, 0x80000000, 0x3F800000, 0xBF800000, 0x40000000]
        rnd = lambda: int(rng.integers(0, 1 << 32))
    return [pal[int(rng.integers(0, len(pal)))] if rng.random() < palette_frac else rnd()
            for _ in range(v)]


def check_select_brute_force(lib=None, trials=400, seed=11):
    """Tiny rows: the oracle's set is the unique subset that holds every
    forced id and whose non-forced members beat every excluded id."""
    rng = np.random.default_rng(seed)
    for trial in range(trials):
        is_bf16 = bool(trial % 2)
        M = int(rng.integers(1, 10))
        nvp = int(rng.integers(0, M + 3))
        v = min(nvp, M)
        I = int(rng.integers(0, 3))
        L = int(rng.integers(0, 3))
        K = int(rng.integers(max(1, I + L), max(1, I + L) + M + 3))
        row = _rand_row_bits(rng, M, is_bf16)
        arr = np.array(row, dtype=np.uint16 if is_bf16 else np.uint32).reshape(1, 1, M)
        got = oracle.topk_select(arr, [nvp], K, I, L, lib=lib)[0, 0]
        n = min(K, v)
        sols = _pins.brute_force_select(row, v, K, I, L, is_bf16)
        assert len(sols) == 1, (trial, row, v, K, I, L, sols)
        assert list(got[:n]) == sols[0], (trial, row, v, K, I, L, list(got), sols)
        assert (got[n:] == -1).all(), (trial, list(got))


def check_select_lexsort_special_case(lib=None, trials=200, seed=12):
    """NaN-free fp32 rows without zeros: selection = numpy lexsort on
    (forced desc, value desc, id asc), then ascending ids."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        M = int(rng.integers(1, 300))
        v = int(rng.integers(0, M + 1))
        I = int(rng.integers(0, 3))
        L = int(rng.integers(0, 4))
        K = int(rng.integers(max(1, I + L), max(I + L, 1) + 40))
        vals = (rng.integers(1, 12, size=M) * rng.choice([-1, 1], size=M)).astype(np.float32)
        arr = vals.reshape(1, 1, M)
        got = oracle.topk_select(arr, [v], K, I, L, lib=lib)[0, 0]
        ids = np.arange(v)
        forced = (ids < I) | (ids >= v - L)
        order = np.lexsort((ids, -vals[:v].astype(np.float64), -forced.astype(np.int64)))
        n = min(K, v)
        want = np.sort(order[:n])
        assert list(got[:n]) == list(want) and (got[n:] == -1).all()


def check_select_short_rows_take_everything(lib=None):
    """v <= K: the selection is every causal block, whatever the scores."""
    rng = np.random.default_rng(4)
    for v in range(0, 17):
        arr = rng.standard_normal((1, 1, 32)).astype(np.float32)
        got = oracle.topk_select(arr, [v], 16, 1, 1, lib=lib)[0, 0]
        assert list(got) == list(range(v)) + [-1] * (16 - v)


def check_select_forced_blocks(lib=None):
    """Init and local blocks are kept even when they hold the lowest scores."""
    M = 40
    vals = np.linspace(1.0, 2.0, M, dtype=np.float32)
    vals[0] = -np.inf
    vals[36:40] = -1e30
    arr = vals.reshape(1, 1, M)
    got = oracle.topk_select(arr, [40], 8, 1, 2, lib=lib)[0, 0]
    # forced: 0 (init), 38, 39 (local); the other 5 are the largest: 31..35
    assert list(got) == [0, 31, 32, 33, 34, 35, 38, 39], list(got)
    got = oracle.topk_select(arr, [37], 8, 2, 1, lib=lib)[0, 0]
    # v = 37: forced 0, 1 and 36; best others 31..35
    assert list(got) == [0, 1, 31, 32, 33, 34, 35, 36], list(got)


def check_select_ties_lower_id(lib=None):
    arr = np.zeros((1, 1, 20), dtype=np.float32)
    got = oracle.topk_select(arr, [20], 4, 0, 0, lib=lib)[0, 0]
    assert list(got) == [0, 1, 2, 3]
    arr[0, 0, 7] = 1.0
    arr[0, 0, 5] = -0.0
    got = oracle.topk_select(arr, [20], 4, 0, 0, lib=lib)[0, 0]
    assert list(got) == [0, 1, 2, 7]


def _fused(flat, seq, dql, K, I, L, table, ts, hs, H, M, lib):
    """The fused oracle on a flat buffer; an error return counts as a
    failed pin (a mutant that breaks the call must not pass silently)."""
    try:
        return oracle.topk_select_sparse_table(flat, seq, dql, K, I, L, table, token_stride=ts,
                                               head_stride=hs, H=H, M=M, lib=lib)
    except ValueError as e:
        raise AssertionError(f"fused oracle rejected a valid call: {e}")


def _fused_layout(rng, B, dql, H, M, is_bf16):
    """A flat score buffer with a capacity-wide head stride and a padded token
    stride.  The tiles between M and the head stride hold +NaN (the largest
    value), so a read past M would change the selection; the buffer has
    spare room at its end so that a layout mistake reads defined memory."""
    T = B * dql
    hs = M + int(rng.integers(0, 10))
    ts = H * hs + int(rng.integers(0, 6))
    n = (T + H + 1) * ts + M
    bits = _rand_row_bits(rng, n, is_bf16, palette_frac=0.3)
    flat = np.array(bits, dtype=np.uint16 if is_bf16 else np.uint32)
    nan = 0x7FC0 if is_bf16 else 0x7FC00000
    for t in range(T):
        for h in range(H):
            base = t * ts + h * hs
            flat[base + M:base + hs] = nan
    return flat, ts, hs


def _seq_lens_mix(rng, B, dql, M):
    """Padded requests, requests shorter than dql, lengths straddling 128-token
    boundaries, and contexts longer than the M-block capacity."""
    out = []
    for _ in range(B):
        kind = int(rng.integers(0, 5))
        if kind == 0:
            out.append(0)
        elif kind == 1:
            out.append(int(rng.integers(1, dql + 1)))
        elif kind == 2:
            out.append(128 * int(rng.integers(1, M + 1)) + int(rng.integers(-dql, dql + 1)))
        elif kind == 3:
            out.append(int(rng.integers(128 * M, 128 * M + 600)))
        else:
            out.append(int(rng.integers(1, 128 * M)))
    return np.maximum(np.array(out, dtype=np.int64), 0).astype(np.int32)


def check_fused_equals_select_then_table(lib=None, trials=60, seed=31):
    """The fused oracle is, by definition ([55235] 实现拆解: the sparse table is
    emitted from the selector's result; [47984] 关键源码片段: row = req * dql +
    local_q), the decode page count, then the selection, then the table.
    Compared element by element with those three pinned steps called one by
    one, on query lengths 1-4, 1-3 heads, capacity-wide and padded score
    layouts, padded and short requests, and block tables narrower than the
    causal range."""
    rng = np.random.default_rng(seed)
    for trial in range(trials):
        is_bf16 = bool(trial % 2)
        dql = int(rng.integers(1, 5))
        H = int(rng.integers(1, 4))
        B = int(rng.integers(1, 7))
        M = int(rng.integers(4, 41))
        I = int(rng.integers(0, 3))
        L = int(rng.integers(0, 3))
        K = int(rng.integers(max(1, I + L), max(1, I + L) + 12))
        flat, ts, hs = _fused_layout(rng, B, dql, H, M, is_bf16)
        seq = _seq_lens_mix(rng, B, dql, M)
        MB = int(rng.integers(1, M + 4))
        table = rng.permutation(1 << 20)[:B * MB].astype(np.int32).reshape(B, MB)
        T = B * dql
        idx, bt, ctx = _fused(flat, seq, dql, K, I, L, table, ts, hs, H, M, lib)
        nvp = oracle.num_valid_pages_decode(seq, dql, lib=lib)
        idx2 = oracle.topk_select(flat, nvp, K, I, L, token_stride=ts, head_stride=hs, T=T, H=H,
                                  M=M, lib=lib)
        bt2, ctx2 = oracle.build_sparse_block_table(idx2, table, seq, dql, lib=lib)
        ctxt = (trial, dql, H, B, M, K, I, L)
        assert (idx == idx2).all(), ("ids", ctxt)
        assert (bt == bt2).all(), ("table", ctxt)
        assert (ctx == ctx2).all(), ("ctx", ctxt)


def check_fused_token_enumeration(lib=None, trials=150, seed=32):
    """Tiny fused calls against an independent formulation: the causal blocks
    are found by listing the query's tokens 0 .. pos one by one, the selection
    by subset enumeration (brute force), and each kept block's table entries
    and ctx by listing its causal tokens and the page-16 pages they fall in."""
    rng = np.random.default_rng(seed)
    for trial in range(trials):
        is_bf16 = bool(trial % 2)
        dql = int(rng.integers(1, 5))
        H = int(rng.integers(1, 4))
        B = int(rng.integers(1, 4))
        M = int(rng.integers(1, 9))
        I = int(rng.integers(0, 3))
        L = int(rng.integers(0, 3))
        K = int(rng.integers(max(1, I + L), max(1, I + L) + 6))
        flat, ts, hs = _fused_layout(rng, B, dql, H, M, is_bf16)
        seq = _seq_lens_mix(rng, B, dql, M)
        MB = int(rng.integers(1, M + 3))
        table = rng.permutation(1 << 20)[:B * MB].astype(np.int32).reshape(B, MB)
        idx, bt, ctx = _fused(flat, seq, dql, K, I, L, table, ts, hs, H, M, lib)
        for req in range(B):
            for q in range(dql):
                row = req * dql + q
                last = int(seq[req]) - dql + q          # query position
                tokens = range(0, last + 1)             # empty when last < 0
                v = min(M, len({x // 128 for x in tokens}))
                for h in range(H):
                    base = row * ts + h * hs
                    bits = [int(b) for b in flat[base:base + M]]
                    sols = _pins.brute_force_select(bits, v, K, I, L, is_bf16)
                    assert len(sols) == 1
                    sel = sols[0]
                    want_idx = sel + [-1] * (K - len(sel))
                    assert list(idx[row, h]) == want_idx, (trial, row, h, list(idx[row, h]),
                                                           want_idx)
                    want_bt = [0] * (8 * K)
                    want_ctx = 0
                    kept = [b for b in sel if b < MB]
                    for j, b in enumerate(kept):
                        mine = [x for x in tokens if x // 128 == b]
                        want_ctx += len(mine)
                        for page in sorted({(x - 128 * b) // 16 for x in mine}):
                            want_bt[8 * j + page] = int(table[req, b]) * 8 + page
                    assert list(bt[row, h]) == want_bt, (trial, row, h)
                    assert int(ctx[row, h]) == want_ctx, (trial, row, h, int(ctx[row, h]),
                                                          want_ctx)


def _index_case(rng, integer_valued):
    """Small decode batch for the index-score oracle: queries [T, H, D],
    pooled keys [NB, D] (bf16), a block table of distinct physical ids with
    some entries out of range, sequence lengths that include padded
    requests and contexts longer than the table."""
    import torch
    dql = int(rng.integers(1, 4))
    B = int(rng.integers(1, 5))
    H = int(rng.integers(1, 4))
    D = int(rng.choice([8, 16, 24]))
    M = int(rng.integers(2, 10))
    MB = int(rng.integers(1, M + 3))
    NB = B * MB + 7
    if integer_valued:
        q = torch.from_numpy(rng.integers(-4, 5, (B * dql, H, D)).astype(np.float32))
        k = torch.from_numpy(rng.integers(-4, 5, (NB, D)).astype(np.float32))
    else:
        q = torch.from_numpy(rng.standard_normal((B * dql, H, D)).astype(np.float32))
        k = torch.from_numpy(rng.standard_normal((NB, D)).astype(np.float32))
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    table = rng.permutation(NB)[:B * MB].astype(np.int32).reshape(B, MB)
    table[rng.random((B, MB)) < 0.1] = NB + 3           # no usable key
    seq = rng.integers(0, 128 * (M + 2), B).astype(np.int32)
    seq[rng.random(B) < 0.2] = 0
    return q, k, table, seq, dql, M


def check_index_scores_against_numpy(lib=None, trials=40, seed=41):
    """The index-score oracle against a vectorised float64 numpy formulation
    (gather the request's keys through the block table, einsum with the
    queries): exact on integer-valued inputs, to 1e-12 relative otherwise;
    NaN past each row's causal count, -inf for causal blocks without a key."""
    rng = np.random.default_rng(seed)
    for trial in range(trials):
        q, k, table, seq, dql, M = _index_case(rng, integer_valued=trial % 2 == 0)
        got = oracle.index_scores(q, k, table, seq, dql, M, lib=lib)
        T, H, D = q.shape
        B, MB = table.shape
        qd = q.float().numpy().astype(np.float64)
        kd = k.float().numpy().astype(np.float64)
        nvp = oracle.num_valid_pages_decode(seq, dql, lib=lib)
        for t in range(T):
            req = t // dql
            v = min(M, int(nvp[t]))
            phys = np.array([table[req, b] if b < MB else -1 for b in range(v)], dtype=np.int64)
            ok = (phys >= 0) & (phys < kd.shape[0])
            keys = kd[np.where(ok, phys, 0)]                              # [v, D]
            want = np.einsum("hd,bd->hb", qd[t], keys)
            want[:, ~ok] = -np.inf
            row = got[t]
            assert np.isnan(row[:, v:]).all(), (trial, t)
            if trial % 2 == 0:
                assert np.array_equal(row[:, :v], want), (trial, t)
            else:
                fin = np.isfinite(want)
                assert np.array_equal(np.isfinite(row[:, :v]), fin), (trial, t)
                assert np.allclose(row[:, :v][fin], want[fin], rtol=1e-12, atol=1e-12), (trial, t)
                assert (row[:, :v][~fin] == -np.inf).all()


def check_index_scores_one_hot(lib=None, trials=30, seed=42):
    """A one-hot query e_j reads coordinate j of the key of the block's
    physical id: score[t, h, b] = k[block_table[req, b], j(t, h)]."""
    import torch
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        q, k, table, seq, dql, M = _index_case(rng, integer_valued=False)
        T, H, D = q.shape
        j = rng.integers(0, D, (T, H))
        oh = np.zeros((T, H, D), dtype=np.float32)
        for t in range(T):
            for h in range(H):
                oh[t, h, j[t, h]] = 1.0
        got = oracle.index_scores(torch.from_numpy(oh).to(torch.bfloat16), k, table, seq, dql, M,
                                  lib=lib)
        kd = k.float().numpy()
        nvp = oracle.num_valid_pages_decode(seq, dql, lib=lib)
        for t in range(T):
            req = t // dql
            for h in range(H):
                for b in range(min(M, int(nvp[t]))):
                    p = int(table[req, b]) if b < table.shape[1] else -1
                    want = kd[p, j[t, h]] if 0 <= p < kd.shape[0] else -np.inf
                    assert got[t, h, b] == want, (t, h, b, got[t, h, b], want)


def _attention_case(rng, G=None, D=None):
    """A small decode batch for the attention oracle: a sparse table built by
    the (pinned) table oracle from random selections, and random bf16 q, k,
    v over a page-16 cache."""
    import torch
    dql = int(rng.integers(1, 4))
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 3))
    G = int(rng.integers(1, 4)) if G is None else G
    D = int(rng.choice([4, 8, 16])) if D is None else D
    K = int(rng.integers(1, 6))
    MB = 6
    seq = rng.integers(0, 128 * MB, B).astype(np.int32)
    seq[rng.random(B) < 0.2] = 0
    ids = rng.integers(-1, MB + 1, (B * dql, H, K)).astype(np.int32)
    NP = B * MB * 8
    table = rng.permutation(B * MB).astype(np.int32).reshape(B, MB)
    bt, ctx = oracle.build_sparse_block_table(ids, table, seq, dql)
    q = torch.from_numpy(rng.standard_normal((B * dql, H, G, D)).astype(np.float32))
    k = torch.from_numpy(rng.standard_normal((NP, 16, H, D)).astype(np.float32))
    v = torch.from_numpy(rng.standard_normal((NP, 16, H, D)).astype(np.float32))
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), bt, ctx


def check_attention_against_numpy(lib=None, trials=30, seed=51):
    """The attention oracle against a vectorised float64 numpy formulation:
    gather the row's ctx tokens through the page-16 table, softmax of the
    scaled dot products, weighted sum of the values; zeros for an empty
    context."""
    rng = np.random.default_rng(seed)
    for _ in range(trials):
        q, k, v, bt, ctx = _attention_case(rng)
        scale = float(rng.uniform(0.05, 1.0))
        got = oracle.sparse_decode_attention(q, k, v, bt, ctx, scale, lib=lib)
        qd = q.float().numpy().astype(np.float64)
        kd = k.float().numpy().astype(np.float64)
        vd = v.float().numpy().astype(np.float64)
        T, H, G, D = qd.shape
        for t in range(T):
            for h in range(H):
                n = int(ctx[t, h])
                if n == 0:
                    assert (got[t, h] == 0).all()
                    continue
                j = np.arange(n)
                pages = bt[t, h][j // 16]
                kj = kd[pages, j % 16, h]                       # [n, D]
                vj = vd[pages, j % 16, h]
                sc = scale * (qd[t, h] @ kj.T)                  # [G, n]
                p = np.exp(sc - sc.max(axis=1, keepdims=True))
                want = (p / p.sum(axis=1, keepdims=True)) @ vj
                assert np.allclose(got[t, h], want, rtol=1e-12, atol=1e-12), (t, h)


def check_attention_closed_forms(lib=None, seed=52):
    """Equal keys give uniform weights, so the output is the mean of the
    context's values; a one-token context returns that token's value
    exactly."""
    import torch
    rng = np.random.default_rng(seed)
    for _ in range(10):
        q, k, v, bt, ctx = _attention_case(rng)
        k = torch.ones_like(k)                          # every key equal
        got = oracle.sparse_decode_attention(q, k, v, bt, ctx, 0.7, lib=lib)
        vd = v.float().numpy().astype(np.float64)
        T, H = ctx.shape
        for t in range(T):
            for h in range(H):
                n = int(ctx[t, h])
                if n == 0:
                    continue
                j = np.arange(n)
                mean = vd[bt[t, h][j // 16], j % 16, h].mean(axis=0)
                assert np.allclose(got[t, h], mean[None, :], rtol=1e-12, atol=1e-12)
        one = np.minimum(ctx, 1).astype(np.int32)
        got = oracle.sparse_decode_attention(q, k, v, bt, one, 0.7, lib=lib)
        for t in range(T):
            for h in range(H):
                if one[t, h]:
                    want = vd[bt[t, h][0], 0, h]
                    assert np.array_equal(got[t, h], np.broadcast_to(want, got[t, h].shape))


ALL_CHECKS = [
    check_total_order_golden,
    check_total_order_exhaustive_bf16,
    check_total_order_random_fp32,
    check_causal_pages_golden,
    check_varlen_prefill_positions,
    check_spec_decode_worked_example,
    check_table_duplicates_ignored,
    check_table_full_selection_covers_causal_len,
    check_table_input_order_irrelevant,
    check_select_brute_force,
    check_select_lexsort_special_case,
    check_select_short_rows_take_everything,
    check_select_forced_blocks,
    check_select_ties_lower_id,
    check_fused_equals_select_then_table,
    check_fused_token_enumeration,
    check_index_scores_against_numpy,
    check_index_scores_one_hot,
    check_attention_against_numpy,
    check_attention_closed_forms,
]
