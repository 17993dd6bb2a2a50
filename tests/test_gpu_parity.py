"""CUDA path vs the CPU oracle, element by element (needs a GB300).

Indices, sparse tables and context lengths are integers: the bar is
bit-exact equality.  Every call goes through the C ABI (via the thin
binding); the oracle only ever sees CPU copies of the same inputs.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu


def _nvp_for(w):
    if w.seq_lens is not None:
        return oracle.num_valid_pages_decode(w.seq_lens.numpy(), w.dql)
    return oracle.num_valid_pages_varlen(w.cu_seqlens_q.numpy(), w.prefix_lens.numpy())


def _prep(w, tail=float("-inf")):
    """Apply the pages' -inf sentinel (or another tail value) beyond each
    token's causal page count, and the planted block; returns the oracle's
    page counts."""
    nvp = _nvp_for(w)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), tail)
    if w.plant_u is not None:
        synth.plant(w.scores, torch.from_numpy(nvp), w.plant_u, w.plant_value)
    return nvp


def _gpu_select(scores_cpu, nvp, K, I, L, dev, M=None):
    s = scores_cpu.to(dev)
    n = torch.from_numpy(np.ascontiguousarray(nvp)).to(dev)
    out = bsa.bsa_topk_select(s, n, K, I, L, M=M)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _assert_equal(got, want, what):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        r = tuple(bad[0][:-1])
        raise AssertionError(f"{what}: {len(bad)} mismatches; first at {tuple(bad[0])}: "
                             f"got {got[r]} want {want[r]}")


# ---------------------------------------------------------------- page counts

@pytest.mark.parametrize("dql", [1, 2, 4, 8])
def test_num_valid_pages_decode(cuda_device, dql):
    g = torch.Generator().manual_seed(100 + dql)
    seq = torch.randint(0, 140000, (333,), generator=g, dtype=torch.int32)
    seq[:10] = torch.tensor([0, 1, 2, 3, 127, 128, 129, 130, 131, 132], dtype=torch.int32)
    got = bsa.bsa_num_valid_pages_decode(seq.to(cuda_device), dql).cpu().numpy()
    _assert_equal(got, oracle.num_valid_pages_decode(seq.numpy(), dql), "decode pages")


def test_num_valid_pages_varlen(cuda_device):
    w = synth.mixed_prefill_decode(seed=41)
    cu, pre = w.cu_seqlens_q, w.prefix_lens
    got = bsa.bsa_num_valid_pages_varlen(cu.to(cuda_device), pre.to(cuda_device), w.T)
    _assert_equal(got.cpu().numpy(), oracle.num_valid_pages_varlen(cu.numpy(), pre.numpy()),
                  "varlen pages")
    # rows outside [cu[0], cu[N]) get 0; chunked prefill with a prefix
    cu2 = torch.tensor([5, 6, 300, 301], dtype=torch.int32)
    pre2 = torch.tensor([1000, 127, 128], dtype=torch.int32)
    got2 = bsa.bsa_num_valid_pages_varlen(cu2.to(cuda_device), pre2.to(cuda_device), 310)
    want2 = np.zeros(310, dtype=np.int32)
    for i in range(3):
        for r in range(int(cu2[i]), int(cu2[i + 1])):
            want2[r] = -(-(int(pre2[i]) + r - int(cu2[i]) + 1) // 128)
    _assert_equal(got2.cpu().numpy(), want2, "varlen pages with offsets")


# ---------------------------------------------------------------- workloads

WORKLOADS = {
    "tiny_decode": lambda: synth.tiny_decode(),
    "short_decode": lambda: synth.short_decode(),
    "long_decode_k16": lambda: synth.long_decode(K=16),
    "long_decode_k64": lambda: synth.long_decode(K=64),
    "mixed_prefill_decode": lambda: synth.mixed_prefill_decode(),
}


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("seed_offset", [0, 1, 2])
def test_select_workloads(cuda_device, name, seed_offset):
    w = WORKLOADS[name]()
    if seed_offset:
        # reseed the score draw, keep the shapes and lengths
        w.scores.copy_(synth.normal_scores(w.scores.shape, w.dtype, 5000 + seed_offset))
        if name == "short_decode":
            synth.inject_specials(w.scores, 6000 + seed_offset)
    nvp = _prep(w)
    want = oracle.topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
    got = _gpu_select(w.scores, nvp, w.K, w.num_init, w.num_local, cuda_device)
    _assert_equal(got, want, name)


@pytest.mark.parametrize("name", ["short_decode", "long_decode_k16", "mixed_prefill_decode"])
def test_select_never_reads_past_causal_bound(cuda_device, name):
    """Tiles beyond the causal page count hold +NaN (the largest value) here
    instead of -inf: the result must not change."""
    w = WORKLOADS[name]()
    nvp = _prep(w, tail=float("nan"))
    want = oracle.topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
    got = _gpu_select(w.scores, nvp, w.K, w.num_init, w.num_local, cuda_device)
    _assert_equal(got, want, name + " with +NaN tail")


# ---------------------------------------------------------------- boundaries

VALID = [0, 1, 2, 3, 15, 16, 17, 63, 64, 65, 73, 74, 75, 127, 128, 129, 255, 256, 257,
         511, 512, 513, 1023, 1024]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [1, 4, 16, 64])
@pytest.mark.parametrize("IL", [(0, 0), (1, 1), (1, 2), (2, 3)])
def test_select_boundary_sweep(cuda_device, dtype, K, IL):
    I, L = IL
    if K < I + L:
        pytest.skip("K < num_init + num_local is rejected by the host")
    M = 1030
    reps = 3
    rows = len(VALID) * reps
    scores = synth.normal_scores((rows, 2, M), dtype, seed=K * 10 + I + 7 * L)
    synth.inject_specials(scores, seed=K + 99, frac_each=0.02, frac_ties=0.05)
    nvp = np.array(VALID * reps, dtype=np.int32)
    synth.fill_tail(scores, torch.from_numpy(nvp), float("-inf"))
    want = oracle.topk_select(scores, nvp, K, I, L)
    got = _gpu_select(scores, nvp, K, I, L, cuda_device)
    _assert_equal(got, want, f"sweep dtype={dtype} K={K} I={I} L={L}")


@pytest.mark.parametrize("dtype,M", [(torch.bfloat16, 74), (torch.bfloat16, 600),
                                     (torch.bfloat16, 1024), (torch.float32, 300),
                                     (torch.float32, 512)])
@pytest.mark.parametrize("K,I,L", [(17, 1, 0), (18, 1, 0), (20, 1, 2), (24, 2, 3), (32, 1, 2),
                                   (32, 0, 0), (5, 1, 2)])
def test_select_pair_path_topk_sweep(cuda_device, dtype, M, K, I, L):
    """The pair path (topk <= 32, rows <= 2 KB) on both sides of K' = 16,
    where the top-16 merges give way to full 32-entry sorts, over row lengths
    from a handful of blocks to the capacity, with NaN / Inf / zero / tie
    specials."""
    assert bsa.bsa_select_policy(10**5, M, K, 0 if dtype == torch.bfloat16 else 1)["path"] == \
        bsa.BSA_PATH_PAIR
    rows = 96
    rng = np.random.default_rng(K * 100 + M)
    nvp = rng.integers(0, M + 40, rows).astype(np.int32)
    nvp[:8] = [0, 1, K - 1, K, K + 1, M, M - 1, 2 * K]
    scores = synth.normal_scores((rows, 2, M), dtype, seed=K * 13 + M)
    synth.inject_specials(scores, seed=K + M, frac_each=0.02, frac_ties=0.05)
    synth.fill_tail(scores, torch.from_numpy(np.minimum(nvp, M)), float("-inf"))
    want = oracle.topk_select(scores, nvp, K, I, L)
    got = _gpu_select(scores, nvp, K, I, L, cuda_device)
    _assert_equal(got, want, f"pair sweep dtype={dtype} M={M} K={K} I={I} L={L}")


@pytest.mark.parametrize("dtype,M", [(torch.bfloat16, 74), (torch.bfloat16, 300),
                                     (torch.bfloat16, 1024), (torch.float32, 200),
                                     (torch.float32, 512)])
@pytest.mark.parametrize("K,I,L", [(33, 1, 1), (40, 0, 0), (48, 1, 2), (61, 2, 3), (64, 1, 2),
                                   (64, 0, 0)])
def test_select_octet_path_topk_sweep(cuda_device, dtype, M, K, I, L):
    """The octet path (32 < topk <= 64, rows <= 2 KB) over row lengths from a
    handful of blocks (every block a candidate) past 128 non-forced blocks
    (threshold from representatives), with NaN / Inf / zero / tie specials,
    in the plain and the fused call."""
    dt = 0 if dtype == torch.bfloat16 else 1
    if K > M:
        pytest.skip("K > M is rejected by the host")
    assert bsa.bsa_select_policy(10**5, M, K, dt)["path"] == bsa.BSA_PATH_OCTET
    rows = 160
    rng = np.random.default_rng(K * 1000 + M + 7 * I + L)
    nvp = rng.integers(0, M + 40, rows).astype(np.int32)
    nvp[:12] = [0, 1, K - 1, K, K + 1, M, M - 1, 2 * K, 128 + I + L, 129 + I + L, 130 + I + L,
                M // 2]
    scores = synth.normal_scores((rows, 2, M), dtype, seed=K * 17 + M)
    synth.inject_specials(scores, seed=K + M + 1, frac_each=0.02, frac_ties=0.05)
    synth.fill_tail(scores, torch.from_numpy(np.minimum(nvp, M)), float("-inf"))
    want = oracle.topk_select(scores, nvp, K, I, L)
    got = _gpu_select(scores, nvp, K, I, L, cuda_device)
    _assert_equal(got, want, f"octet sweep dtype={dtype} M={M} K={K} I={I} L={L}")


@pytest.mark.parametrize("bf16", [True, False])
def test_fused_octet_path(cuda_device, bf16):
    """The fused call at topk 64 on the octet path: ids, table and ctx."""
    dtype = torch.bfloat16 if bf16 else torch.float32
    w = synth.fused_table(seed=91, B=200, dql=2, H=2, M=1024 if bf16 else 512, K=64,
                          dtype=dtype)
    synth.inject_specials(w.scores, seed=92, frac_each=0.005, frac_ties=0.02)
    nvp = _prep(w)
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, w.K, 1, 2, w.block_table.numpy())
    dev = cuda_device
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(
        w.scores.to(dev), w.seq_lens.to(dev), w.dql, w.K, 1, 2, w.block_table.to(dev))
    torch.cuda.synchronize()
    _assert_equal(idx.cpu().numpy(), want_idx, "fused octet idx")
    _assert_equal(bt.cpu().numpy(), want_bt, "fused octet table")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "fused octet ctx")
    del nvp


@pytest.mark.parametrize("M", [16, 74, 128, 129, 256, 257, 512, 513, 1024])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_select_capacity_boundaries(cuda_device, M, dtype):
    """Capacities around the launch policy's boundaries, all rows full."""
    T, H, K = 40, 3, 16
    scores = synth.normal_scores((T, H, M), dtype, seed=M)
    synth.inject_specials(scores, seed=M + 1)
    nvp = np.full(T, M + 5, dtype=np.int32)   # clamps to M
    nvp[::7] = np.arange(len(nvp[::7])) % (M + 1)
    want = oracle.topk_select(scores, nvp, K, 1, 1)
    got = _gpu_select(scores, nvp, K, 1, 1, cuda_device)
    _assert_equal(got, want, f"capacity M={M}")


ADVERSARIAL = ["equal", "ascending", "descending", "all_nan", "all_neg_inf", "signed_zeros",
               "negative_only", "neg_nan_payloads", "few_positive", "blocks_of_ties"]


def _adversarial_row(kind, M, rng, bf16):
    if kind == "equal":
        x = np.full(M, 0.75, np.float32)
    elif kind == "ascending":
        x = np.linspace(-3, 3, M).astype(np.float32)
    elif kind == "descending":
        x = np.linspace(3, -3, M).astype(np.float32)
    elif kind == "all_nan":
        x = np.full(M, np.nan, np.float32)
    elif kind == "all_neg_inf":
        x = np.full(M, -np.inf, np.float32)
    elif kind == "signed_zeros":
        x = np.where(rng.random(M) < 0.5, -0.0, 0.0).astype(np.float32)
    elif kind == "negative_only":
        x = -np.abs(rng.standard_normal(M)).astype(np.float32) - 0.01
    elif kind == "neg_nan_payloads":
        x = np.full(M, -1.0, np.float32)
    elif kind == "few_positive":
        x = -np.abs(rng.standard_normal(M)).astype(np.float32)
        x[rng.integers(0, M, 5)] = 1.0
    else:  # blocks_of_ties
        x = np.repeat(rng.integers(-3, 4, M // 8 + 1), 8)[:M].astype(np.float32)
    t = torch.from_numpy(x)
    t = t.to(torch.bfloat16) if bf16 else t
    if kind == "neg_nan_payloads":
        bits = t.view(torch.int16 if bf16 else torch.int32)
        base = 0xFF80 if bf16 else 0xFF800000
        width = 1 << (16 if bf16 else 32)
        for i in range(0, M, 3):
            v = base | (1 + (i * 7919) % (0x7F if bf16 else 0x7FFFFF))
            bits[i] = v - width
    return t


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("M", [100, 700, 3000])
def test_select_adversarial_rows(cuda_device, bf16, M):
    rng = np.random.default_rng(M)
    rows = [_adversarial_row(k, M, rng, bf16) for k in ADVERSARIAL]
    scores = torch.stack(rows).view(len(rows), 1, M)
    for K, I, L in [(16, 1, 1), (64, 1, 2), (5, 0, 0)]:
        nvp = np.array([M] * len(rows), dtype=np.int32)
        want = oracle.topk_select(scores, nvp, K, I, L)
        got = _gpu_select(scores, nvp, K, I, L, cuda_device)
        _assert_equal(got, want, f"adversarial bf16={bf16} M={M} K={K}")


@pytest.mark.parametrize("bf16", [True, False])
@pytest.mark.parametrize("want_idx", [True, False])
def test_fused_adversarial_rows(cuda_device, bf16, want_idx):
    """The fused call on rows that overflow any fixed candidate list (ties,
    NaN runs) or hold only negative scores: overflowing rows are finished by
    the fix-up launch, which also writes their table and ctx."""
    M = 500
    rng = np.random.default_rng(11)
    rows = [_adversarial_row(k, M, rng, bf16) for k in ADVERSARIAL] * 3
    T = len(rows)
    scores = torch.stack(rows).view(T, 1, M)
    seq = np.full(T, M * 128, dtype=np.int32)
    seq[len(ADVERSARIAL):2 * len(ADVERSARIAL)] -= 777        # partial last block
    seq[2 * len(ADVERSARIAL):] = rng.integers(2000, M * 128, len(ADVERSARIAL))
    table = synth.random_block_table(T, M, seed=5)
    want_idx_np, want_bt, want_ctx = oracle.topk_select_sparse_table(
        scores, seq, 1, 16, 1, 2, table.numpy())
    dev = cuda_device
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(
        scores.to(dev), torch.from_numpy(seq).to(dev), 1, 16, 1, 2, table.to(dev),
        want_idx=want_idx)
    torch.cuda.synchronize()
    if want_idx:
        _assert_equal(idx.cpu().numpy(), want_idx_np, "fused adversarial idx")
    _assert_equal(bt.cpu().numpy(), want_bt, "fused adversarial table")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "fused adversarial ctx")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_select_all_negative_long_rows(cuda_device, dtype):
    """Long-context rows whose scores are all negative, with one planted
    block that is the least negative: the threshold works in key space for
    rows of any sign."""
    w = synth.long_decode(seed=21, B=96, H=2, M=1024 if dtype == torch.bfloat16 else 512,
                          K=16, dtype=dtype)
    nvp = _nvp_for(w)
    w.scores.copy_(-(w.scores.float().abs() + 0.25).to(dtype))
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    synth.plant(w.scores, torch.from_numpy(nvp), w.plant_u, -0.01)
    want = oracle.topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
    got = _gpu_select(w.scores, nvp, w.K, w.num_init, w.num_local, cuda_device)
    _assert_equal(got, want, f"all-negative rows {dtype}")


# ---------------------------------------------------------------- layouts

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_select_strided_and_misaligned_views(cuda_device, dtype):
    """A capacity-8192 buffer used with M=300 (head stride 8192), and views
    whose rows start off 16-byte boundaries."""
    T, H, cap, M, K = 50, 3, 8192, 300, 16
    big = synth.normal_scores((T, H, cap), dtype, seed=77)
    synth.inject_specials(big, seed=78)
    nvp = (np.arange(T, dtype=np.int32) * 37) % 320
    want = oracle.topk_select(big[:, :, :M].contiguous(), nvp, K, 1, 2)
    dev_big = big.to(cuda_device)
    out = bsa.bsa_topk_select(dev_big, torch.from_numpy(nvp).to(cuda_device), K, 1, 2, M=M)
    torch.cuda.synchronize()
    _assert_equal(out.cpu().numpy(), want, "capacity-strided view")
    # odd element offsets and an odd row stride
    for off in (1, 3, 5):
        flat = synth.normal_scores((T * H * 301 + 16,), dtype, seed=off)
        view_cpu = flat[off:off + T * H * 301].view(T, H, 301)[:, :, :M]
        want = oracle.topk_select(view_cpu.contiguous(), nvp, K, 1, 2)
        dflat = flat.to(cuda_device)
        dview = dflat[off:off + T * H * 301].view(T, H, 301)[:, :, :M]
        out = bsa.bsa_topk_select(dview, torch.from_numpy(nvp).to(cuda_device), K, 1, 2)
        torch.cuda.synchronize()
        _assert_equal(out.cpu().numpy(), want, f"misaligned view offset {off}")


# ---------------------------------------------------------------- split rows

@pytest.mark.parametrize("M", [2000, 4096, 8192])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [16, 64])
def test_select_split_rows(cuda_device, M, dtype, K):
    """Few long rows: the policy splits each row over several warps and the
    last-arriving warp merges.  Run twice: the tickets must reset."""
    T, H = 24, 2
    pol = bsa.bsa_select_policy(T * H, M, K, bsa.BSA_DTYPE_BF16 if dtype == torch.bfloat16
                                else bsa.BSA_DTYPE_FP32,
                                torch.cuda.get_device_properties(cuda_device).multi_processor_count)
    assert pol["chunks_per_row"] > 1, pol
    scores = synth.normal_scores((T, H, M), dtype, seed=M + K)
    synth.inject_specials(scores, seed=M + K + 1)
    nvp = np.linspace(0, M + 10, T).astype(np.int32)
    want = oracle.topk_select(scores, nvp, K, 1, 2)
    for _ in range(2):
        got = _gpu_select(scores, nvp, K, 1, 2, cuda_device)
        _assert_equal(got, want, f"split M={M} K={K}")


def test_select_split_graph_replay(cuda_device):
    """CUDA-graph capture of the split path, replayed on fresh inputs."""
    T, H, M, K = 16, 2, 8192, 16
    dev = cuda_device
    nvp = np.linspace(1, M, T).astype(np.int32)
    s_dev = torch.empty((T, H, M), dtype=torch.bfloat16, device=dev)
    n_dev = torch.from_numpy(nvp).to(dev)
    out = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    s_dev.copy_(synth.normal_scores((T, H, M), torch.bfloat16, seed=1).to(dev))
    bsa.bsa_topk_select(s_dev, n_dev, K, 1, 1, out_idx=out)  # warm-up (workspace)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            bsa.bsa_topk_select(s_dev, n_dev, K, 1, 1, out_idx=out)
    for rep in range(3):
        scores = synth.normal_scores((T, H, M), torch.bfloat16, seed=10 + rep)
        s_dev.copy_(scores.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        _assert_equal(out.cpu().numpy(), oracle.topk_select(scores, nvp, K, 1, 1),
                      f"graph replay {rep}")


# ---------------------------------------------------------------- sparse table

def test_sparse_table_worked_example(cuda_device):
    """The speculative-decode example printed in the vLLM PR #47984 report."""
    import json
    import os
    from tests.conftest import GOLDEN
    with open(os.path.join(GOLDEN, "spec_decode_sparse_table.json")) as f:
        ex = json.load(f)
    idx = torch.tensor(ex["topk_idx"], dtype=torch.int32).view(12, 1, 4).to(cuda_device)
    bt, ctx = bsa.bsa_build_sparse_block_table(
        idx, torch.tensor(ex["block_table"], dtype=torch.int32).to(cuda_device),
        torch.tensor(ex["seq_lens"], dtype=torch.int32).to(cuda_device), ex["decode_query_len"])
    torch.cuda.synchronize()
    assert list(ctx.cpu().numpy()[:, 0]) == ex["expected_ctx"]
    for r, pref in enumerate(ex["expected_bt_nonzero_prefix"]):
        assert list(bt.cpu().numpy()[r, 0]) == pref + [0] * (ex["row_width"] - len(pref))


@pytest.mark.parametrize("H,K,dql", [(1, 16, 4), (2, 16, 1), (3, 7, 3), (1, 64, 2), (2, 300, 1),
                                     (2, 32, 2), (1, 13, 1), (4, 1, 1), (3, 17, 2), (1, 33, 1),
                                     (2, 47, 3), (3, 63, 1), (1, 65, 2)])
def test_sparse_table_random_ids(cuda_device, H, K, dql):
    """Arbitrary ids: -1, out-of-range, beyond the block table, duplicates."""
    g = torch.Generator().manual_seed(K * 31 + H)
    B, MB = 97, 40
    seq = torch.randint(0, 6000, (B,), generator=g, dtype=torch.int32)
    seq[::9] = 0
    seq[1::11] = 1
    T = B * dql
    idx = torch.randint(-3, 60, (T, H, K), generator=g, dtype=torch.int32)
    idx[:, :, 1::4] = idx[:, :, ::4][:, :, :idx[:, :, 1::4].shape[2]]  # duplicates
    table = synth.random_block_table(B, MB, seed=K)
    want_bt, want_ctx = oracle.build_sparse_block_table(idx.numpy(), table.numpy(),
                                                        seq.numpy(), dql)
    bt, ctx = bsa.bsa_build_sparse_block_table(idx.to(cuda_device), table.to(cuda_device),
                                               seq.to(cuda_device), dql)
    torch.cuda.synchronize()
    _assert_equal(bt.cpu().numpy(), want_bt, "sparse table")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "sparse ctx")


@pytest.mark.parametrize("K", [33, 48, 64])
@pytest.mark.parametrize("pattern", ["distinct", "all_same", "descending", "mixed"])
def test_sparse_table_warp_row_patterns(cuda_device, K, pattern):
    """Topk between 33 and 64 (one warp per row, two ids per lane): ids all
    distinct, all one id, in descending order, or distinct with -1 holes and
    repeats, against the oracle."""
    g = torch.Generator().manual_seed(900 + K)
    B, H, dql, MB = 150, 2, 2, 128
    seq = torch.randint(0, 128 * MB + 300, (B,), generator=g, dtype=torch.int32)
    seq[::13] = 0
    T = B * dql
    rows = T * H
    if pattern == "distinct":
        idx = torch.stack([torch.randperm(MB, generator=g)[:K] for _ in range(rows)])
    elif pattern == "all_same":
        idx = torch.randint(0, 40, (rows, 1), generator=g).expand(rows, K).clone()
    elif pattern == "descending":
        idx = torch.arange(K - 1, -1, -1).expand(rows, K).clone() + torch.randint(
            0, MB - K, (rows, 1), generator=g)
    else:
        idx = torch.stack([torch.randperm(MB, generator=g)[:K] for _ in range(rows)])
        idx[:, ::7] = -1
        idx[:, 5::9] = idx[:, 4::9][:, :idx[:, 5::9].shape[1]]
    idx = idx.to(torch.int32).view(T, H, K)
    table = synth.random_block_table(B, MB, seed=K + 7)
    want_bt, want_ctx = oracle.build_sparse_block_table(idx.numpy(), table.numpy(),
                                                        seq.numpy(), dql)
    bt, ctx = bsa.bsa_build_sparse_block_table(idx.to(cuda_device), table.to(cuda_device),
                                               seq.to(cuda_device), dql)
    torch.cuda.synchronize()
    _assert_equal(bt.cpu().numpy(), want_bt, f"sparse table {pattern}")
    _assert_equal(ctx.cpu().numpy(), want_ctx, f"sparse ctx {pattern}")


@pytest.mark.parametrize("K", [16, 32, 64])
@pytest.mark.parametrize("offset_words", [1, 4])
def test_sparse_table_unaligned_output_and_many_rows(cuda_device, K, offset_words):
    """An output table that starts 4 or 16 bytes past a 32-byte boundary takes
    the element-wise store form; 12000 rows span many grid strides."""
    g = torch.Generator().manual_seed(500 + K)
    B, H, dql, MB = 3000, 2, 2, 64
    seq = torch.randint(0, 8200, (B,), generator=g, dtype=torch.int32)
    T = B * dql
    idx = torch.randint(-2, 70, (T, H, K), generator=g, dtype=torch.int32)
    idx[:, :, 3::5] = idx[:, :, ::5][:, :, :idx[:, :, 3::5].shape[2]]
    table = synth.random_block_table(B, MB, seed=K + 1)
    want_bt, want_ctx = oracle.build_sparse_block_table(idx.numpy(), table.numpy(), seq.numpy(), dql)
    n = T * H * K * 8
    flat = torch.full((n + 8,), -7, dtype=torch.int32, device=cuda_device)
    bt = flat[offset_words:offset_words + n].view(T, H, K * 8)
    assert bt.data_ptr() % 32 == 4 * offset_words
    _, ctx = bsa.bsa_build_sparse_block_table(idx.to(cuda_device), table.to(cuda_device),
                                              seq.to(cuda_device), dql, sparse_bt=bt)
    torch.cuda.synchronize()
    _assert_equal(bt.cpu().numpy(), want_bt, "sparse table (unaligned)")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "sparse ctx")
    assert int(flat[0].item()) == -7 and int(flat[-1].item()) == -7


@pytest.mark.parametrize("variant", ["as_given", "dql1_h2", "fp32_small_table", "no_idx"])
def test_fused_select_sparse_table(cuda_device, variant):
    kw = {}
    if variant == "dql1_h2":
        kw = dict(B=300, dql=1, H=2, M=600)
    elif variant == "fp32_small_table":
        kw = dict(B=64, dql=3, H=1, M=200, dtype=torch.float32, max_len=40000)
    w = synth.fused_table(**kw)
    table = w.block_table
    if variant == "fp32_small_table":
        table = table[:, :150].contiguous()  # narrower than some causal ranges
    synth.inject_specials(w.scores, seed=3)
    nvp = _prep(w)
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, w.K, w.num_init, w.num_local, table.numpy())
    dev = cuda_device
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(
        w.scores.to(dev), w.seq_lens.to(dev), w.dql, w.K, w.num_init, w.num_local,
        table.to(dev), want_idx=variant != "no_idx")
    torch.cuda.synchronize()
    if variant != "no_idx":
        _assert_equal(idx.cpu().numpy(), want_idx, "fused idx")
    _assert_equal(bt.cpu().numpy(), want_bt, "fused table")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "fused ctx")
    # the unfused GPU pipeline gives the same result
    n = bsa.bsa_num_valid_pages_decode(w.seq_lens.to(dev), w.dql)
    i2 = bsa.bsa_topk_select(w.scores.to(dev), n, w.K, w.num_init, w.num_local)
    b2, c2 = bsa.bsa_build_sparse_block_table(i2, table.to(dev), w.seq_lens.to(dev), w.dql)
    torch.cuda.synchronize()
    _assert_equal(b2.cpu().numpy(), want_bt, "unfused table")
    _assert_equal(c2.cpu().numpy(), want_ctx, "unfused ctx")


@pytest.mark.parametrize("offset_words", [1, 4])
def test_fused_table_output_off_32_byte_boundary(cuda_device, offset_words):
    """The fused call writes 32-byte table slots with one 256-bit store when
    the table is 32-byte aligned; tables 4 or 16 bytes past a boundary take
    the element-wise path and give the same result."""
    w = synth.fused_table(B=96, dql=2, H=2, M=300)
    table = w.block_table
    nvp = _prep(w)
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, w.K, w.num_init, w.num_local, table.numpy())
    dev = cuda_device
    T, H, K = w.T, w.H, w.K
    flat = torch.full((T * H * K * 8 + 8,), -9, dtype=torch.int32, device=dev)
    bt = flat[offset_words:offset_words + T * H * K * 8].view(T, H, K * 8)
    assert bt.data_ptr() % 32 == 4 * offset_words
    idx, bt_out, ctx = bsa.bsa_topk_select_sparse_table(
        w.scores.to(dev), w.seq_lens.to(dev), w.dql, K, w.num_init, w.num_local, table.to(dev),
        sparse_bt=bt)
    torch.cuda.synchronize()
    assert bt_out.data_ptr() == bt.data_ptr()
    _assert_equal(idx.cpu().numpy(), want_idx, "fused idx (offset table)")
    _assert_equal(bt.cpu().numpy(), want_bt, "fused table (offset)")
    _assert_equal(ctx.cpu().numpy(), want_ctx, "fused ctx (offset table)")
    assert int(flat[0].item()) == -9 and int(flat[-1].item()) == -9
    del nvp


def test_fused_long_rows_split(cuda_device):
    """Fused path on few long rows (split + merge + table epilogue)."""
    w = synth.fused_table(B=8, dql=2, H=2, M=8192, max_len=8192 * 128)
    nvp = _prep(w)
    assert nvp.max() > 4096
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, w.K, 1, 1, w.block_table.numpy())
    dev = cuda_device
    for _ in range(2):
        idx, bt, ctx = bsa.bsa_topk_select_sparse_table(
            w.scores.to(dev), w.seq_lens.to(dev), w.dql, w.K, 1, 1, w.block_table.to(dev))
        torch.cuda.synchronize()
        _assert_equal(idx.cpu().numpy(), want_idx, "fused split idx")
        _assert_equal(bt.cpu().numpy(), want_bt, "fused split table")
        _assert_equal(ctx.cpu().numpy(), want_ctx, "fused split ctx")


# ---------------------------------------------------------------- errors

def test_host_rejects_bad_arguments(cuda_device):
    s = torch.zeros((4, 1, 32), dtype=torch.float32, device=cuda_device)
    n = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    for K, I, L, code in [(0, 0, 0, -3), (33, 0, 0, -3), (2, 2, 1, -3), (1025, 0, 0, -3)]:
        with pytest.raises(bsa.BsaError) as e:
            bsa.bsa_topk_select(s, n, K, I, L)
        assert e.value.status == code
    with pytest.raises(ValueError):
        bsa.bsa_topk_select(s.to(torch.float16), n, 4, 1, 1)
    idx = torch.zeros((5, 1, 4), dtype=torch.int32, device=cuda_device)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_build_sparse_block_table(idx, torch.zeros((2, 3), dtype=torch.int32,
                                                          device=cuda_device),
                                         torch.zeros(2, dtype=torch.int32, device=cuda_device), 2)
    assert e.value.status == -6


# ---------------------------------------------------------------- full size

@pytest.mark.parametrize("K", [16, 64])
def test_full_size_bench_workload_sampled(cuda_device, K):
    """The benchmark's workload at full size (131072 requests, 2 heads, 1024
    tiles, topk 16 and 64) in the benchmark's launch configuration: every row
    is checked for the properties any correct answer has, and a random sample
    of token rows is compared with the oracle element by element."""
    dev = cuda_device
    # the benchmark's workload (synth.long_decode with 131072 requests, its
    # block table) with the -inf tail and the planted block placed by the
    # oracle's page counts
    w = synth.long_decode(seed=1003, device=dev, B=131072, H=2, M=1024, K=K,
                          dtype=torch.bfloat16)
    nvp_host = oracle.num_valid_pages_decode(w.seq_lens.cpu().numpy(), w.dql)
    nvp = torch.from_numpy(nvp_host).to(dev)
    synth.fill_tail(w.scores, nvp, float("-inf"))
    synth.plant(w.scores, nvp, w.plant_u, w.plant_value)
    table = synth.random_block_table(w.B, w.M, seed=2003, device=dev)
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(w.scores, w.seq_lens, w.dql, w.K,
                                                    w.num_init, w.num_local, table)
    torch.cuda.synchronize()
    K = w.K
    v = torch.clamp(nvp.long(), max=w.M).view(-1, 1, 1)
    n = torch.clamp(v, max=K)
    slot = torch.arange(K, device=dev).view(1, 1, K)
    valid = slot < n
    assert torch.equal(idx[~valid.expand_as(idx)], torch.full_like(idx[~valid.expand_as(idx)], -1))
    assert bool(((idx < v) | ~valid).all())
    asc = (idx[:, :, 1:] > idx[:, :, :-1]) | ~valid[:, :, 1:]
    assert bool(asc.all())
    assert bool((idx[:, :, 0] == 0).all())                     # init block
    assert bool((idx[:, :, K - 1] == v[:, :, 0] - 1).all())    # local blocks
    assert bool((idx[:, :, K - 2] == v[:, :, 0] - 2).all())
    # every row: a valid selection, including the exchange property
    from tests import _props
    _props.check_selection(w.scores, nvp, idx, K, w.num_init, w.num_local)
    # sampled rows against the oracle
    g = torch.Generator().manual_seed(11)
    rows = torch.randperm(w.T, generator=g)[:3000].sort().values
    sc = w.scores[rows.to(dev)].cpu()
    seq = w.seq_lens[rows.to(dev)].cpu().numpy()
    tb = table[rows.to(dev)].cpu().numpy()
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(sc, seq, 1, K, w.num_init,
                                                                  w.num_local, tb)
    r = rows.to(dev)
    _assert_equal(idx[r].cpu().numpy(), want_idx, "full-size sampled idx")
    _assert_equal(bt[r].cpu().numpy(), want_bt, "full-size sampled table")
    _assert_equal(ctx[r].cpu().numpy(), want_ctx, "full-size sampled ctx")
    # the unfused selector agrees on every row
    idx2 = bsa.bsa_topk_select(w.scores, nvp, K, w.num_init, w.num_local)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)
