"""Sparse decode attention over the page-16 table (needs a GB300).

The consumer of the selector's sparse table (vLLM PR #47984 report, 实现拆解
items 1-2; vLLM PR #47502 report, 实现拆解 item 5), under the readings pinned
on the CPU in the oracle.  The table fed to both sides is the oracle's; the
GPU's own fused select + table is checked to give the same table, so the
three steps (select, table, attention) agree end to end.

Tolerance: the kernel works in fp32.  A score is a dot product of D bf16
values scaled by 1/sqrt(D) (error about D * 2^-24 * sum |q k| * scale, below
1e-4 here) and an output is a convex combination of at most K * 128 value
rows accumulated in fp32 (error about ctx * 2^-24 * max |v|, below 6e-4 for
2048 tokens of N(0, 1) values); 1e-3 absolute covers both.
"""
import math

import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.mark.parametrize("B,dql,H,G,D,MB,K", [
    (24, 2, 2, 3, 128, 96, 16),     # GQA group of 3, two index/KV heads
    (16, 1, 1, 8, 64, 200, 64),     # topk 64, group of 8
    (32, 4, 1, 1, 256, 40, 16),     # query length 4, one query head, wide heads
    (20, 4, 1, 4, 64, 64, 16),      # the bench's shape: group of 4, D = 64
    (16, 2, 2, 2, 128, 80, 32),     # group of 2, D = 128
    (12, 1, 3, 1, 64, 50, 16),      # one query head, three KV heads
])
def test_sparse_decode_attention(cuda_device, B, dql, H, G, D, MB, K):
    dev = cuda_device
    seed = B + MB + K
    g = torch.Generator().manual_seed(seed)
    seq = torch.randint(1, MB * 128 + 1, (B,), generator=g, dtype=torch.int32)
    seq[::7] = 0                                            # padded requests
    table = synth.paged_block_table(B, MB, B * MB, seed=seed + 1)
    T = B * dql
    scores = synth.normal_scores((T, H, MB), torch.bfloat16, seed=seed + 2)
    nvp = oracle.num_valid_pages_decode(seq.numpy(), dql)
    synth.fill_tail(scores, torch.from_numpy(nvp), float("-inf"))
    idx, bt, ctx = oracle.topk_select_sparse_table(scores, seq.numpy(), dql, K, 1, 1,
                                                   table.numpy())
    num_pages = B * MB * 8
    q = synth.normal_scores((T, H, G, D), torch.bfloat16, seed=seed + 3)
    k = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=seed + 4)
    v = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=seed + 5)
    scale = 1.0 / math.sqrt(D)
    want = oracle.sparse_decode_attention(q, k, v, bt, ctx, scale)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    got = bsa.bsa_sparse_decode_attention(qd, kd, vd, torch.from_numpy(bt).to(dev),
                                          torch.from_numpy(ctx).to(dev))
    torch.cuda.synchronize()
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert err.max() <= TOL, f"max error {err.max()}"
    assert (got.cpu().numpy()[ctx == 0] == 0).all(), "empty contexts must give zeros"
    # end to end: the GPU's fused select + table gives the oracle's table,
    # so attention over it is the same computation
    _, bt2, ctx2 = bsa.bsa_topk_select_sparse_table(scores.to(dev), seq.to(dev), dql, K, 1, 1,
                                                    table.to(dev), want_idx=False)
    torch.cuda.synchronize()
    assert np.array_equal(bt2.cpu().numpy(), bt) and np.array_equal(ctx2.cpu().numpy(), ctx)
    got2 = bsa.bsa_sparse_decode_attention(qd, kd, vd, bt2, ctx2)
    torch.cuda.synchronize()
    assert torch.equal(got2, got)


@pytest.mark.parametrize("G", [2, 8])
def test_sparse_decode_attention_pages_out_of_range(cuda_device, G):
    """Tokens on page ids outside the cache take no part, as in the oracle;
    a row whose every page is out of range yields zeros."""
    dev = cuda_device
    T, H, D, K = 6, 1, 64, 2
    num_pages = 5
    bt = np.zeros((T, H, K * 8), dtype=np.int32)
    bt[:, 0, :4] = [[1, 7, 2, -1], [0, 1, 2, 3], [9, 9, 9, 9], [4, 4, 5, 0],
                    [3, -2, 1, 2], [2, 2, 2, 2]]
    ctx = np.array([[50], [64], [40], [33], [64], [1]], dtype=np.int32)
    q = synth.normal_scores((T, H, G, D), torch.bfloat16, seed=1)
    k = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=2)
    v = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=3)
    want = oracle.sparse_decode_attention(q, k, v, bt, ctx, 0.125)
    got = bsa.bsa_sparse_decode_attention(q.to(dev), k.to(dev), v.to(dev),
                                          torch.from_numpy(bt).to(dev),
                                          torch.from_numpy(ctx).to(dev), scale=0.125)
    torch.cuda.synchronize()
    assert np.abs(got.cpu().numpy() - want).max() <= TOL
    assert (got.cpu().numpy()[2] == 0).all()


def test_sparse_decode_attention_rejects_bad_arguments(cuda_device):
    dev = cuda_device
    q = torch.zeros((2, 1, 9, 64), dtype=torch.bfloat16, device=dev)      # G = 9 > 8
    k = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16, device=dev)
    bt = torch.zeros((2, 1, 8), dtype=torch.int32, device=dev)
    ctx = torch.zeros((2, 1), dtype=torch.int32, device=dev)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_sparse_decode_attention(q, k, k, bt, ctx)
    assert e.value.status == -2
    q = torch.zeros((2, 1, 2, 96), dtype=torch.bfloat16, device=dev)      # D = 96
    k = torch.zeros((4, 16, 1, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_sparse_decode_attention(q, k, k, bt, ctx)
    assert e.value.status == -2
