"""CUDA-graph capture of the calls a decode step makes (needs a GB300).

The header states that every call except the allocation-free selector can
be captured in a CUDA graph.  Each call here is captured once and replayed on
fresh inputs written into the captured buffers; every replay is compared with
the oracle on those inputs."""
import math

import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu


def _capture(fn, dev):
    fn()                                   # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            fn()
    torch.cuda.synchronize()
    return graph


@pytest.mark.parametrize("K", [16, 64])
def test_graph_fused_select_table(cuda_device, K):
    dev = cuda_device
    B, dql, H, M = 96, 2, 2, 1024
    w = synth.fused_table(seed=70 + K, B=B, dql=dql, H=H, M=M, K=K)
    s_dev = w.scores.to(dev)
    seq_dev = w.seq_lens.to(dev)
    tab_dev = w.block_table.to(dev)
    idx = torch.empty((B * dql, H, K), dtype=torch.int32, device=dev)
    bt = torch.empty((B * dql, H, K * 8), dtype=torch.int32, device=dev)
    ctx = torch.empty((B * dql, H), dtype=torch.int32, device=dev)

    def fn():
        bsa.bsa_topk_select_sparse_table(s_dev, seq_dev, dql, K, 1, 2, tab_dev, out_idx=idx,
                                         sparse_bt=bt, sparse_ctx=ctx)

    graph = _capture(fn, dev)
    for rep in range(3):
        scores = synth.normal_scores((B * dql, H, M), torch.bfloat16, seed=700 + rep)
        nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), dql)
        synth.fill_tail(scores, torch.from_numpy(nvp), float("-inf"))
        s_dev.copy_(scores.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
            scores, w.seq_lens.numpy(), dql, K, 1, 2, w.block_table.numpy())
        assert np.array_equal(idx.cpu().numpy(), want_idx), rep
        assert np.array_equal(bt.cpu().numpy(), want_bt), rep
        assert np.array_equal(ctx.cpu().numpy(), want_ctx), rep


def test_graph_index_score_and_attention(cuda_device):
    """A decode step's tail as one graph: index scores + selection + table,
    then attention over the table; replayed on fresh queries."""
    dev = cuda_device
    B, dql, H, D, M, K, G, Da = 24, 2, 2, 64, 300, 16, 2, 64
    g = np.random.default_rng(3)
    seq = torch.from_numpy(g.integers(1, M * 128 + 1, B).astype(np.int32))
    nb = B * M
    table = synth.paged_block_table(B, M, nb, seed=4)
    _, k = synth.index_inputs(5, B * dql, H, D, nb, integer_valued=True)
    kc = synth.normal_scores((nb * 8, 16, H, Da), torch.bfloat16, seed=6)
    vc = synth.normal_scores((nb * 8, 16, H, Da), torch.bfloat16, seed=7)
    T = B * dql
    q_dev = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    qa_dev = torch.empty((T, H, G, Da), dtype=torch.bfloat16, device=dev)
    scores = torch.full((T, H, M), float("-inf"), dtype=torch.float32, device=dev)
    idx = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    bt = torch.empty((T, H, K * 8), dtype=torch.int32, device=dev)
    ctx = torch.empty((T, H), dtype=torch.int32, device=dev)
    out = torch.empty((T, H, G, Da), dtype=torch.float32, device=dev)
    k_dev, kc_dev, vc_dev = k.to(dev), kc.to(dev), vc.to(dev)
    seq_dev, tab_dev = seq.to(dev), table.to(dev)

    def fn():
        bsa.bsa_index_score_topk_select(q_dev, k_dev, tab_dev, seq_dev, dql, K, 1, 1, M=M,
                                        scores=scores, out_idx=idx, sparse_bt=bt,
                                        sparse_ctx=ctx)
        bsa.bsa_sparse_decode_attention(qa_dev, kc_dev, vc_dev, bt, ctx, out=out)

    q0, _ = synth.index_inputs(8, T, H, D, 1, integer_valued=True)
    q_dev.copy_(q0.to(dev))
    qa_dev.copy_(synth.normal_scores((T, H, G, Da), torch.bfloat16, seed=9).to(dev))
    graph = _capture(fn, dev)
    nvp = oracle.num_valid_pages_decode(seq.numpy(), dql)
    for rep in range(2):
        q, _ = synth.index_inputs(20 + rep, T, H, D, 1, integer_valued=True)
        qa = synth.normal_scores((T, H, G, Da), torch.bfloat16, seed=30 + rep)
        q_dev.copy_(q.to(dev))
        qa_dev.copy_(qa.to(dev))
        graph.replay()
        torch.cuda.synchronize()
        want_s = oracle.index_scores(q, k, table.numpy(), seq.numpy(), dql, M)
        s32 = np.where(np.isnan(want_s), -np.inf, want_s).astype(np.float32)
        want_idx = oracle.topk_select(s32, nvp, K, 1, 1)
        want_bt, want_ctx = oracle.build_sparse_block_table(want_idx, table.numpy(), seq.numpy(),
                                                            dql)
        assert np.array_equal(idx.cpu().numpy(), want_idx), rep
        assert np.array_equal(bt.cpu().numpy(), want_bt), rep
        assert np.array_equal(ctx.cpu().numpy(), want_ctx), rep
        want_att = oracle.sparse_decode_attention(qa, kc, vc, want_bt, want_ctx,
                                                  1.0 / math.sqrt(Da))
        assert np.abs(out.cpu().numpy() - want_att).max() <= 1e-3, rep
