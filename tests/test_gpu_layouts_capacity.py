"""Output layouts and the capture-time capacity (needs a GB300).

* Head-major output: the vLLM PR #49149 report (实现拆解 items 1-2) keeps
  Triton consumers on an [H, T, K] buffer and hands the token-major producer
  a transpose(0, 1) view; the selector writes through any such strided view.
* Prefill-heavy unified batches at the 8192-tile capacity: the vLLM PR
  #47502 report (关键源码片段, indexer_msa.py) freezes the unified buffer at
  [*, H, 8192] and serves decode rows [:nd] and prefill rows [nd:] in one
  call.  Thousands of rows of up to 8192 blocks take the unsplit row path.

Every result is compared element by element with the oracle (all rows where
the oracle finishes in seconds, a seeded sample of rows otherwise) and, at
full size, every row is checked for the properties any correct answer has.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth
from tests import _props

pytestmark = pytest.mark.gpu


def _eq(got, want, what):
    got = np.asarray(got)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        raise AssertionError(f"{what}: {len(bad)} mismatches; first at {tuple(bad[0])}")


def _decode_case(name):
    if name == "pair":
        w = synth.short_decode(seed=61)
    elif name == "row64":
        w = synth.long_decode(seed=62, B=96, H=3, K=64)
    else:  # split: few long rows
        w = synth.long_decode(seed=63, B=24, H=2, M=8192, K=16, min_len=300000,
                              max_len=8192 * 128)
    nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), w.dql)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    if w.plant_u is not None:
        synth.plant(w.scores, torch.from_numpy(nvp), w.plant_u, w.plant_value)
    return w, nvp


@pytest.mark.parametrize("name", ["pair", "row64", "split"])
@pytest.mark.parametrize("layout", ["head_major", "padded"])
def test_select_into_strided_output(cuda_device, name, layout):
    """The selector writes into a transpose(0, 1) view of a head-major
    [H, T, K] buffer, or into a token-major buffer with padded rows; the
    padding is left untouched."""
    w, nvp = _decode_case(name)
    T, H, K = w.T, w.H, w.K
    want = oracle.topk_select(w.scores, nvp, K, w.num_init, w.num_local)
    dev = cuda_device
    if layout == "head_major":
        buf = torch.full((H, T, K), -7, dtype=torch.int32, device=dev)
        view = buf.transpose(0, 1)
    else:
        buf = torch.full((T, H, K + 5), -7, dtype=torch.int32, device=dev)
        view = buf[:, :, :K]
    out = bsa.bsa_topk_select(w.scores.to(dev), torch.from_numpy(nvp).to(dev), K, w.num_init,
                              w.num_local, out_idx=view)
    torch.cuda.synchronize()
    assert out.data_ptr() == view.data_ptr()
    _eq(view.cpu().numpy(), want, f"{name} {layout}")
    if layout == "head_major":
        _eq(buf.cpu().numpy(), want.transpose(1, 0, 2), f"{name} head-major buffer")
    else:
        assert bool((buf[:, :, K:] == -7).all()), "padding was written"


@pytest.mark.parametrize("K", [16, 64])
def test_fused_into_head_major_ids(cuda_device, K):
    """The fused call writes its ids head-major while the sparse table and
    ctx stay token-major."""
    w = synth.fused_table(seed=64, B=80, dql=3, H=2, M=400, K=K)
    nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), w.dql)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
        w.scores, w.seq_lens.numpy(), w.dql, K, w.num_init, w.num_local, w.block_table.numpy())
    dev = cuda_device
    buf = torch.full((w.H, w.T, K), -7, dtype=torch.int32, device=dev)
    _, bt, ctx = bsa.bsa_topk_select_sparse_table(
        w.scores.to(dev), w.seq_lens.to(dev), w.dql, K, w.num_init, w.num_local,
        w.block_table.to(dev), out_idx=buf.transpose(0, 1))
    torch.cuda.synchronize()
    _eq(buf.transpose(0, 1).cpu().numpy(), want_idx, "fused head-major ids")
    _eq(bt.cpu().numpy(), want_bt, "fused table")
    _eq(ctx.cpu().numpy(), want_ctx, "fused ctx")


def _prefill_heavy(dtype, dev, seed):
    """32 decode rows with contexts up to 1M tokens, then two 8192-token
    prefill chunks: one from position 0 (1..64 blocks), one at the end of a
    1M-token context (8129..8192 blocks); 4 index heads in a [16416, 4, 8192]
    buffer (the capture-time capacity)."""
    M = 8192
    w = synth.mixed_prefill_decode(seed=seed, device=dev, H=4, M=M, K=16, dtype=dtype,
                                   prefill_prefix=(0, M * 128 - 8192),
                                   decode_max_prefix=M * 128 - 1)
    nvp_host = oracle.num_valid_pages_varlen(w.cu_seqlens_q.cpu().numpy(),
                                             w.prefix_lens.cpu().numpy())
    nvp = torch.from_numpy(nvp_host).to(dev)
    synth.fill_tail(w.scores, nvp, float("-inf"))
    synth.inject_specials(w.scores, seed=seed + 1, frac_each=0.002, frac_ties=0.01)
    return w, nvp_host, nvp


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("K,L", [(16, 1), (64, 2)])
def test_prefill_heavy_batch_at_full_capacity(cuda_device, dtype, K, L):
    dev = cuda_device
    w, nvp_host, nvp = _prefill_heavy(dtype, dev, seed=70 + K)
    T, H, M = w.T, w.H, w.M
    dt = bsa.BSA_DTYPE_BF16 if dtype == torch.bfloat16 else bsa.BSA_DTYPE_FP32
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    pol = bsa.bsa_select_policy(T * H, M, K, dt, sms)
    assert pol["chunks_per_row"] == 1, "thousands of rows must not take the split path"
    # rows within 2 KB on the pair / octet path, the rest on the wide path
    assert pol["path"] == (bsa.BSA_PATH_PAIR if K <= 32 else bsa.BSA_PATH_OCTET)
    assert pol["long_rows"] == 1
    out = bsa.bsa_topk_select(w.scores, nvp, K, 1, L)
    torch.cuda.synchronize()
    _props.check_selection(w.scores, nvp, out, K, 1, L)
    # element by element on a seeded sample: every decode row, the first and
    # last rows of each prefill, and 1500 random rows
    g = torch.Generator().manual_seed(K)
    nd = w.notes["num_decode"]
    pick = set(range(nd)) | {nd, nd + 8191, nd + 8192, T - 1}
    pick |= set(torch.randint(0, T, (1500,), generator=g).tolist())
    rows = torch.tensor(sorted(pick), dtype=torch.int64)
    sc = w.scores[rows.to(dev)].cpu()
    want = oracle.topk_select(sc, nvp_host[rows.numpy()], K, 1, L)
    _eq(out[rows.to(dev)].cpu().numpy(), want, f"prefill-heavy {dtype} K={K}")
    # and the same answer from a second call (no state carried between calls)
    out2 = bsa.bsa_topk_select(w.scores, nvp, K, 1, L)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)
