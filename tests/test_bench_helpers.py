"""bench.py's algorithmic byte count against a hand-computed example (the
definition the roofline uses: the non-forced causal prefix of each row when
the row needs a selection, the id write, the page-count read, and for the
fused call the block-table gathers, the table and ctx writes)."""
import os
import sys
from types import SimpleNamespace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_hand_example():
    sys.path.insert(0, ROOT)
    import bench
    w = SimpleNamespace(K=4, H=2, num_init=1, num_local=1, dtype=torch.bfloat16, M=10, T=3)
    # page counts 0, 3, 12 -> v = 0, 3, 10; only the last row has v > K
    b = bench.algorithmic_bytes(w, np.array([0, 3, 12], dtype=np.int32), "fused")
    # scores: (10 - 2 forced) bf16 x 2 heads = 32 B; ids 3*2*4*4 = 96 B; page counts 3*4 = 12 B
    assert b["score_read"] == 32
    assert b["select"] == 32 + 96 + 12
    # gathers: n = 0 + 3 + 4 ids per head x 2 heads x 4 B = 56 B
    # table + ctx: 3 tokens x 2 heads x (4*8*4 + 4) = 792 B
    assert b["fused"] == 140 + 56 + 792
    assert b["table_builder"] == 96 + 12 + 56 + 792
    assert b["per_row_fused"] == (140 + 56 + 792) / 6


def test_roofline_kernel_and_traffic_follow_the_policy():
    """The bench names the selector kernel the launch policy picks, and takes
    committed ncu traffic only for the kernel, topk and request count it was
    captured on."""
    sys.path.insert(0, ROOT)
    import bench
    import block_sparse_attention_topk_gb300 as bsa
    rows = 131072 * 2
    p16 = bsa.bsa_select_policy(rows, 1024, 16, bsa.BSA_DTYPE_BF16, 152)
    p64 = bsa.bsa_select_policy(rows, 1024, 64, bsa.BSA_DTYPE_BF16, 152)
    assert bench.KERNEL_OF_PATH[p16["path"]] == "pair_select_kernel"
    assert bench.KERNEL_OF_PATH[p64["path"]] == "octet_select_kernel"
    assert bench.dominant_kernel(p64["path"], True).startswith("octet_select_kernel (fused")
    import json
    import tempfile
    ent = {"kernel": "pair_select_kernel<bf16, topk<=16>", "topk": 16, "requests": 131072,
           "dram_bytes_per_launch": 1}
    with tempfile.TemporaryDirectory() as d:
        f = os.path.join(d, "traffic.json")
        for sha, ok in ((bench.select_source_sha(), True), ("0" * 16, False)):
            with open(f, "w") as fh:
                json.dump({p: dict(ent, source_sha=sha) for p in ("fused", "unfused")}, fh)
            for path in ("fused", "unfused"):
                got = bench.read_traffic(path, "pair_select_kernel", 16, 131072, f)
                assert (got is not None) == ok, "traffic is used only for the current source"
                assert bench.read_traffic(path, "select_kernel", 64, 131072, f) is None
                assert bench.read_traffic(path, "pair_select_kernel", 32, 131072, f) is None
                assert bench.read_traffic(path, "pair_select_kernel", 16, 65536, f) is None


def test_index_score_bytes_hand_example():
    """The fused index score + select's byte count: queries, the table
    entries and keys of each request's causal blocks, the causal scores of
    each row, sequence lengths and ids."""
    sys.path.insert(0, ROOT)
    import bench
    seq = np.array([0, 200, 129], dtype=np.int32)    # 0, 2, 2 causal blocks
    b = bench.index_score_bytes(seq, 1, 2, 8, 4, 3, valid_blocks=3)
    q = 3 * 2 * 8 * 2                 # [T, H, D] bf16
    table = 4 * 4                     # 4 causal blocks
    keys = 3 * 8 * 2                  # 3 usable keys of D bf16
    scores = (0 + 2 + 2) * 2 * 4      # causal entries x heads x fp32
    assert b == q + table + keys + scores + 3 * 4 + 3 * 2 * 3 * 4


def test_attention_bytes_hand_example():
    """Sparse attention bytes: key and value rows of every context token,
    table entries and ctx, queries in and outputs out."""
    sys.path.insert(0, ROOT)
    import bench
    ctx = np.array([[0], [100]], dtype=np.int32)        # 2 rows, H = 1
    b = bench.attention_bytes(ctx, 1, 2, 64, 4)
    kv = 100 * 64 * 2 * 2
    table = 2 * (4 * 8 * 4 + 4)
    qo = 2 * 2 * 64 * (2 + 4)
    assert b == kv + table + qo
