"""The device status word (needs a GB300).

With a word registered, the kernels set BSA_STATUS_* bits when they meet a
block-table entry, page id or context length that the calls handle without a
fault but that is not valid, and their outputs stay what the plain
computation gives: where the oracle defines that result (a -1 entry expands
to page ids -8 + p; an out-of-range page takes no part; a context past the
table is clamped) the outputs are compared with it.  Valid inputs leave the
word at 0, and with no word registered nothing is recorded.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture
def word(cuda_device):
    w = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    bsa.bsa_set_status_word(w)
    yield w
    bsa.bsa_set_status_word(None, cuda_device)


def _workload(K, M=512, B=64, dql=2, H=2, seed=300):
    w = synth.fused_table(seed=seed + K, device="cpu", B=B, dql=dql, H=H, M=M, K=K)
    nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), dql)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    return w


def _fused(w, dev, table):
    return bsa.bsa_topk_select_sparse_table(w.scores.to(dev), w.seq_lens.to(dev), w.dql, w.K,
                                            w.num_init, w.num_local, table.to(dev))


@pytest.mark.parametrize("K", [16, 64, 128])   # pair, octet and row paths; seg, seg64, generic builders
def test_valid_inputs_leave_status_clear(cuda_device, word, K):
    dev = cuda_device
    w = _workload(K)
    idx, bt, ctx = _fused(w, dev, w.block_table)
    bsa.bsa_build_sparse_block_table(idx, w.block_table.to(dev), w.seq_lens.to(dev), w.dql)
    assert bsa.bsa_read_status() == 0


@pytest.mark.parametrize("K", [16, 64, 128])
def test_negative_block_id_is_reported(cuda_device, word, K):
    """Block 0 (always kept: num_init = 1) of some requests maps to -1."""
    dev = cuda_device
    w = _workload(K)
    table = w.block_table.clone()
    table[::3, 0] = -1
    idx, bt, ctx = _fused(w, dev, table)
    assert bsa.bsa_read_status() & bsa.BSA_STATUS_BAD_BLOCK_ID
    ref_idx, ref_bt, ref_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, K, w.num_init, w.num_local, table.numpy())
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(bt.cpu().numpy(), ref_bt)
    assert np.array_equal(ctx.cpu().numpy(), ref_ctx)
    # the standalone builder reports the same entries
    assert bsa.bsa_read_status() == 0
    bt2, ctx2 = bsa.bsa_build_sparse_block_table(idx, table.to(dev), w.seq_lens.to(dev), w.dql)
    assert bsa.bsa_read_status() & bsa.BSA_STATUS_BAD_BLOCK_ID
    assert np.array_equal(bt2.cpu().numpy(), ref_bt)
    assert np.array_equal(ctx2.cpu().numpy(), ref_ctx)


@pytest.mark.parametrize("K", [16, 64])
def test_block_id_limit(cuda_device, word, K):
    """BSA_MAX_PHYS_BLOCK is the largest id whose page ids fit int32."""
    dev = cuda_device
    w = _workload(K)
    r = int(np.argmax(w.seq_lens.numpy() > 0))       # a request whose block 0 is kept
    table = w.block_table.clone()
    table[r, 0] = 0x0FFFFFFF
    idx, bt, ctx = _fused(w, dev, table)
    assert bsa.bsa_read_status() == 0
    ref = oracle.topk_select_sparse_table(w.scores, w.seq_lens.numpy(), w.dql, K, w.num_init,
                                          w.num_local, table.numpy())
    assert np.array_equal(bt.cpu().numpy(), ref[1])
    assert (bt.cpu().numpy()[r * w.dql] == 0x7FFFFFF8).any()
    table[r, 0] = 0x10000000
    _fused(w, dev, table)
    assert bsa.bsa_read_status() == bsa.BSA_STATUS_BAD_BLOCK_ID


@pytest.mark.parametrize("D", [128, 96])   # segment and thread scoring
def test_index_score_missing_keys_are_reported(cuda_device, word, D):
    dev = cuda_device
    B, dql, H, M, K = 24, 1, 2, 200, 16
    seq = torch.full((B,), M * 128, dtype=torch.int32)
    nb = B * M
    q, k = synth.index_inputs(5, B * dql, H, D, nb)
    clean = synth.paged_block_table(B, M, nb, seed=6)
    bsa.bsa_index_score_topk_select(q.to(dev), k.to(dev), clean.to(dev), seq.to(dev), dql, K, 1, 1,
                                    M=M)
    assert bsa.bsa_read_status() == 0
    narrow = clean[:, :M // 2].contiguous()          # blocks past the table: not an error
    bsa.bsa_index_score_topk_select(q.to(dev), k.to(dev), narrow.to(dev), seq.to(dev), dql, K, 1,
                                    1, M=M)
    assert bsa.bsa_read_status() == 0
    bad = synth.paged_block_table(B, M, nb, seed=6, frac_missing=0.02)
    bsa.bsa_index_score_topk_select(q.to(dev), k.to(dev), bad.to(dev), seq.to(dev), dql, K, 1, 1,
                                    M=M)
    assert bsa.bsa_read_status() == bsa.BSA_STATUS_BAD_BLOCK_ID


def test_attention_bad_page_and_context_are_reported(cuda_device, word):
    dev = cuda_device
    B, dql, H, G, D, M, K = 8, 2, 1, 2, 64, 64, 16
    w = _workload(K, M=M, B=B, dql=dql, H=H, seed=900)
    _, bt, ctx = oracle.topk_select_sparse_table(w.scores, w.seq_lens.numpy(), dql, K, 1, 1,
                                                 w.block_table.numpy())
    npages = B * M * 8
    q = synth.normal_scores((B * dql, H, G, D), torch.bfloat16, seed=1)
    kc = synth.normal_scores((npages, 16, H, D), torch.bfloat16, seed=2)
    vc = synth.normal_scores((npages, 16, H, D), torch.bfloat16, seed=3)

    def run(bt, ctx):
        out = bsa.bsa_sparse_decode_attention(q.to(dev), kc.to(dev), vc.to(dev),
                                              torch.from_numpy(bt).to(dev),
                                              torch.from_numpy(ctx).to(dev))
        ref = oracle.sparse_decode_attention(q, kc, vc, bt, ctx, 1.0 / D ** 0.5)
        assert np.abs(out.cpu().numpy() - ref).max() < 1e-3
        return bsa.bsa_read_status()

    assert run(bt, ctx) == 0
    r = int(np.argmax(ctx.reshape(-1) > 0))
    bad = bt.copy()
    bad.reshape(-1, K * 8)[r, 0] = npages                 # the row's first page: out of range
    assert run(bad, ctx) == bsa.BSA_STATUS_BAD_PAGE
    over = ctx.copy()
    over.reshape(-1)[r] = K * 128 + 5
    assert run(bt, over) == bsa.BSA_STATUS_BAD_CONTEXT
    neg = ctx.copy()
    neg.reshape(-1)[r] = -3
    assert run(bt, neg) == bsa.BSA_STATUS_BAD_CONTEXT


def test_no_word_registered_records_nothing(cuda_device):
    dev = cuda_device
    bsa.bsa_set_status_word(None, dev)
    w = _workload(16)
    table = w.block_table.clone()
    table[:, 0] = -1
    _fused(w, dev, table)
    assert bsa.bsa_read_status() == 0


def test_graph_keeps_the_word_registered_at_capture(cuda_device, word):
    dev = cuda_device
    w = _workload(16)
    table = w.block_table.clone()
    table[::2, 0] = -1
    scores, seq, tab = w.scores.to(dev), w.seq_lens.to(dev), table.to(dev)
    bt = torch.empty((w.T, w.H, 16 * 8), dtype=torch.int32, device=dev)
    ctx = torch.empty((w.T, w.H), dtype=torch.int32, device=dev)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):                       # warm-up outside the capture
        bsa.bsa_topk_select_sparse_table(scores, seq, w.dql, 16, 1, 1, tab, want_idx=False,
                                         sparse_bt=bt, sparse_ctx=ctx)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    word.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bsa.bsa_topk_select_sparse_table(scores, seq, w.dql, 16, 1, 1, tab, want_idx=False,
                                         sparse_bt=bt, sparse_ctx=ctx)
    torch.cuda.synchronize(dev)
    word.zero_()
    g.replay()
    torch.cuda.synchronize(dev)
    assert int(word.item()) == bsa.BSA_STATUS_BAD_BLOCK_ID


def test_long_rows_report_bad_block_ids(cuda_device, word):
    """A 2048-tile buffer with enough rows for the pair path and its list of
    long rows: a -1 entry for block 0 of requests whose rows exceed 2 KB is
    reported by the wide path's table epilogue, and the outputs match the
    oracle."""
    dev = cuda_device
    dql, H, M, K = 1, 2, 2048, 16
    B = (32 * torch.cuda.get_device_properties(dev).multi_processor_count + 255) // H
    g = torch.Generator().manual_seed(3)
    seq = torch.randint(1, M * 128 + 1, (B,), generator=g, dtype=torch.int32)
    table = synth.paged_block_table(B, M, B * M, seed=4)
    long_req = torch.nonzero(seq > 1100 * 128).flatten()[:40]
    table[long_req, 0] = -1
    scores = synth.normal_scores((B * dql, H, M), torch.bfloat16, seed=5, device=dev)
    nvp = oracle.num_valid_pages_decode(seq.numpy(), dql)
    synth.fill_tail(scores, torch.from_numpy(nvp).to(dev), float("-inf"))
    pol = bsa.bsa_select_policy(B * dql * H, M, K, bsa.BSA_DTYPE_BF16,
                                torch.cuda.get_device_properties(dev).multi_processor_count)
    assert pol["long_rows"] == 1
    idx, bt, ctx = bsa.bsa_topk_select_sparse_table(scores, seq.to(dev), dql, K, 1, 2,
                                                    table.to(dev))
    assert bsa.bsa_read_status() == bsa.BSA_STATUS_BAD_BLOCK_ID
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(scores.cpu(), seq.numpy(), dql,
                                                                  K, 1, 2, table.numpy())
    assert np.array_equal(idx.cpu().numpy(), want_idx)
    assert np.array_equal(bt.cpu().numpy(), want_bt)
    assert np.array_equal(ctx.cpu().numpy(), want_ctx)
