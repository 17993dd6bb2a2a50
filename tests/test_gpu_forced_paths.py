"""The group path (4 lanes per row), the octet path (8 lanes per row), the
wide path (one warp per row, bf16 calls) and the row path (one warp per row)
for topk <= 32, forced with BSA_SELECT_PATH,
against the oracle.  The library reads the variable once per process, so
each path runs in a child process."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import oracle
import synth
import block_sparse_attention_topk_gb300 as bsa

want_path = {code}
dev = torch.device("cuda:0")
assert bsa.bsa_select_policy(4096, 1024, 16, 0, 152)["path"] == want_path

def nvp_for(w):
    if w.seq_lens is not None:
        return oracle.num_valid_pages_decode(w.seq_lens.numpy(), w.dql)
    return oracle.num_valid_pages_varlen(w.cu_seqlens_q.numpy(), w.prefix_lens.numpy())

for name, w in (("short_decode", synth.short_decode()),
                ("long_decode", synth.long_decode(B=48, K=16)),
                ("mixed_prefill_decode", synth.mixed_prefill_decode())):
    nvp = nvp_for(w)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    if w.plant_u is not None:
        synth.plant(w.scores, torch.from_numpy(nvp), w.plant_u, w.plant_value)
    want = oracle.topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
    got = bsa.bsa_topk_select(w.scores.to(dev), torch.from_numpy(nvp).to(dev), w.K,
                              w.num_init, w.num_local)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want), name

w = synth.fused_table(B=64)
nvp = nvp_for(w)
synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
want_idx, want_bt, want_ctx = oracle.topk_select_sparse_table(
    w.scores, w.seq_lens.numpy(), w.dql, w.K, w.num_init, w.num_local, w.block_table.numpy())
idx, bt, ctx = bsa.bsa_topk_select_sparse_table(
    w.scores.to(dev), w.seq_lens.to(dev), w.dql, w.K, w.num_init, w.num_local,
    w.block_table.to(dev))
torch.cuda.synchronize()
assert np.array_equal(idx.cpu().numpy(), want_idx), "fused idx"
assert np.array_equal(bt.cpu().numpy(), want_bt), "fused table"
assert np.array_equal(ctx.cpu().numpy(), want_ctx), "fused ctx"
print("ok")
'''


@pytest.mark.gpu
@pytest.mark.parametrize("path,code", [("group", 2), ("row", 0), ("octet", 4), ("wide", 5)])
def test_forced_path_matches_oracle(cuda_device, path, code):
    env = dict(os.environ, BSA_SELECT_PATH=path)
    res = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, code=code)], env=env,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout + res.stderr
