"""bf16 and fp32 buffers wider than 2 KB with topk <= 64 and more than num_sms * 16
rows (needs a GB300): the launch policy sends them to the pair or octet path,
which takes every row whose non-forced range fits in 2 KB and lists the
others for a second launch, the wide path (one warp per row).  Every row is
compared with the oracle element by element: ids for the plain select, ids,
table and context lengths for the fused call; a graph replay and the
allocation-free entry point run the same two launches.  The rows cover:
  * rows of at most 256 non-forced blocks (every element is a candidate) and
    longer rows (a threshold from the representatives first);
  * capacity-wide views whose rows start off a 32-byte boundary (edge chunks
    inside and at the ends of the buffer);
  * NaN, +-Inf, +-0 and exact ties; rows of one repeated value, whose
    candidates overflow the 256-entry list and are redone on the row path;
  * rows that fit in 2 KB (pair / octet path) and longer ones (wide path);
  * topk 1, 16, 33 and 64.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu


def _rows_for_wide(dev):
    return 32 * torch.cuda.get_device_properties(dev).multi_processor_count


def _scores(T, H, width, seed, dev, dtype=torch.bfloat16):
    """N(0, 1) [T, H, width] with specials and ties, and every 97th row one
    repeated value (ties everywhere)."""
    sc = synth.normal_scores((T, H, width), dtype, seed, dev)
    synth.inject_specials(sc, seed=seed + 1, frac_each=0.002, frac_ties=0.02)
    flat = sc.view(T * H, width)
    flat[::97] = 0.75
    return sc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K,I,L", [(1, 0, 0), (16, 1, 2), (33, 1, 1), (64, 1, 2)])
@pytest.mark.parametrize("M,pad", [(2048, 0), (8192, 8), (1500, 5)])
def test_wide_select_matches_oracle(cuda_device, K, I, L, M, pad, dtype):
    dev = cuda_device
    H = 2
    T = (_rows_for_wide(dev) + 255) // H
    g = np.random.default_rng(M + K + pad)
    # valid counts: short rows (every element a candidate), rows just past
    # 256 non-forced blocks, and rows up to the capacity
    nvp_host = g.integers(0, M + 1, T).astype(np.int32)
    nvp_host[::5] = g.integers(0, 300, len(nvp_host[::5]))
    nvp_host[1::11] = 256 + I + L + g.integers(0, 3, len(nvp_host[1::11]))
    nvp_host[2::13] = M
    big = _scores(T, H, M + pad, seed=M + K, dev=dev, dtype=dtype)
    scores = big[:, :, :M]                       # rows start off 32-byte boundaries when pad > 0
    nvp = torch.from_numpy(nvp_host).to(dev)
    synth.fill_tail(scores, nvp, float("-inf"))
    dt = bsa.BSA_DTYPE_BF16 if dtype == torch.bfloat16 else bsa.BSA_DTYPE_FP32
    pol = bsa.bsa_select_policy(T * H, M, K, dt,
                                torch.cuda.get_device_properties(dev).multi_processor_count)
    assert pol["path"] in (bsa.BSA_PATH_PAIR, bsa.BSA_PATH_OCTET) and pol["long_rows"] == 1
    got = bsa.bsa_topk_select(scores, nvp, K, I, L)
    torch.cuda.synchronize()
    want = oracle.topk_select(scores.cpu(), nvp_host, K, I, L)
    bad = np.nonzero((got.cpu().numpy() != want).any(axis=2))
    assert bad[0].size == 0, f"{bad[0].size} rows differ, first (t, h) = {bad[0][0]}, {bad[1][0]}"


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K", [16, 64])
def test_wide_fused_table_matches_oracle(cuda_device, K, dtype):
    """Decode rows of a 2048-tile buffer through the fused select + table."""
    dev = cuda_device
    dql, H, M = 2, 2, 2048
    B = (_rows_for_wide(dev) + 255) // (dql * H)
    g = torch.Generator().manual_seed(K)
    seq = torch.randint(1, M * 128 + 1, (B,), generator=g, dtype=torch.int32)
    seq[::9] = 0                                                # padded requests
    seq[1::7] = torch.randint(1, 300 * 128, (len(seq[1::7]),), generator=g, dtype=torch.int32)
    table = synth.paged_block_table(B, M, B * M, seed=K + 3)
    T = B * dql
    scores = _scores(T, H, M, seed=K + 5, dev=dev, dtype=dtype)
    nvp = oracle.num_valid_pages_decode(seq.numpy(), dql)
    synth.fill_tail(scores, torch.from_numpy(nvp).to(dev), float("-inf"))
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(scores, seq.to(dev), dql, K, 1, 2,
                                                    table.to(dev))
    torch.cuda.synchronize()
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(scores.cpu(), seq.numpy(), dql,
                                                                  K, 1, 2, table.numpy())
    assert np.array_equal(idx.cpu().numpy(), want_idx)
    assert np.array_equal(bt.cpu().numpy(), want_bt)
    assert np.array_equal(ctx.cpu().numpy(), want_ctx)


def test_long_rows_graph_replay_and_noalloc(cuda_device):
    """The memset of the list counter and the two launches replay in a CUDA
    graph (twice, with new scores in between), and the allocation-free entry
    point takes the list from its scratch."""
    dev = cuda_device
    H, M, K = 2, 4096, 16
    T = (_rows_for_wide(dev) + 511) // H
    g = np.random.default_rng(5)
    nvp_host = g.integers(0, M + 1, T).astype(np.int32)
    nvp_host[::3] = g.integers(0, 1000, len(nvp_host[::3]))
    nvp = torch.from_numpy(nvp_host).to(dev)
    scores = _scores(T, H, M, seed=41, dev=dev)
    synth.fill_tail(scores, nvp, float("-inf"))
    out = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    ws = torch.empty(bsa.bsa_topk_workspace_bytes(T, H, M, K, bsa.BSA_DTYPE_BF16, dev),
                     dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        bsa.bsa_topk_select(scores, nvp, K, 1, 2, out_idx=out, workspace=ws)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        bsa.bsa_topk_select(scores, nvp, K, 1, 2, out_idx=out, workspace=ws)
    for seed in (42, 43):
        scores.copy_(_scores(T, H, M, seed=seed, dev=dev))
        synth.fill_tail(scores, nvp, float("-inf"))
        out.fill_(-7)
        graph.replay()
        torch.cuda.synchronize(dev)
        want = oracle.topk_select(scores.cpu(), nvp_host, K, 1, 2)
        assert np.array_equal(out.cpu().numpy(), want), f"graph replay, scores seed {seed}"
    got = bsa.bsa_topk_select_noalloc(scores, nvp, K, 1, 2)
    torch.cuda.synchronize(dev)
    assert np.array_equal(got.cpu().numpy(), want), "allocation-free entry point"
