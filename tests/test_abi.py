"""The C ABI without a GPU: the library builds and loads, exports every
symbol the header declares, and its host-side logic (argument checks, the
launch policy and its capacity boundaries) behaves as documented.  No call
here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bsa_topk.h")


@pytest.fixture(scope="module")
def bsa():
    from block_sparse_attention_topk_gb300 import build
    build.build()
    import block_sparse_attention_topk_gb300 as m
    m.lib()
    return m


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_names(bsa):
    assert _declared() == sorted(bsa.EXPORTED)


def test_library_exports_every_declared_symbol(bsa):
    L = ctypes.CDLL(bsa.library_path())
    for name in _declared():
        assert hasattr(L, name), f"{name} not exported"


def test_library_is_built_for_sm103a(bsa):
    from block_sparse_attention_topk_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def test_status_strings(bsa):
    L = bsa.lib()
    for code in range(-8, 1):
        s = L.bsa_status_string(code).decode()
        assert s and s != "unknown status"


def _policy(bsa, rows, M, K, dtype, sms=152):
    return bsa.bsa_select_policy(rows, M, K, dtype, sms)


BF, FP = 0, 1


@pytest.mark.parametrize("M,dtype,K,path", [
    # pair path: topk <= 32 and a row of at most 2 KB
    (16, FP, 4, 3), (74, BF, 16, 3), (128, BF, 16, 3), (129, BF, 16, 3), (1024, BF, 16, 3),
    (1025, BF, 16, 3), (512, FP, 16, 3), (513, FP, 16, 3), (1024, BF, 32, 3),
    # octet path: 32 < topk <= 64 and a row of at most 2 KB
    (1024, BF, 33, 4), (74, BF, 64, 4), (1024, BF, 64, 4), (512, FP, 64, 4), (513, FP, 64, 4),
    # rows of more than 2 KB, topk <= 64, many rows: the pair / octet path,
    # with the rows over 2 KB left to the wide path
    (1025, BF, 64, 4), (8192, BF, 16, 3), (8192, BF, 1, 3), (65536, BF, 64, 4),
    (8192, FP, 16, 3), (8192, FP, 64, 4),
    # row path: topk > 64
    (1024, BF, 65, 0), (8192, BF, 65, 0), (8192, FP, 65, 0)])
def test_policy_path(bsa, M, dtype, K, path):
    assert _policy(bsa, 10**6, M, K, dtype)["path"] == path


@pytest.mark.parametrize("M,dtype,nv", [
    (74, BF, 1), (128, BF, 1), (129, BF, 1), (256, BF, 1), (257, BF, 2),
    (512, BF, 2), (513, BF, 4), (1024, BF, 4), (8192, BF, 4),
    (74, FP, 1), (128, FP, 1), (129, FP, 2), (256, FP, 2), (257, FP, 4), (1024, FP, 4)])
def test_policy_vectors_per_lane_warp_path(bsa, M, dtype, nv):
    """Warp path (topk 65): vectors per lane per pass switch at 32 lanes x
    16 bytes x {1, 2}: bf16 at 256/257 and 512/513, fp32 at 128/129 and
    256/257."""
    p = _policy(bsa, 1000, M, 65, dtype)
    assert p["path"] in (0, 1) and p["vecs_per_lane"] == nv


def test_policy_production_capacity(bsa):
    """The production 8k+1k graph (74 blocks, query length 4, topk 16) and
    every capacity up to 128 run on the pair path; at topk 64 they run on the
    octet path, never split."""
    for M in (65, 74, 128):
        for rows in (4, 64 * 4 * 4, 10**6):
            p = _policy(bsa, rows, M, 16, BF)
            assert p["path"] == bsa.BSA_PATH_PAIR and p["chunks_per_row"] == 1
            p = _policy(bsa, rows, M, 64, BF)
            assert p["path"] == bsa.BSA_PATH_OCTET and p["chunks_per_row"] == 1


@pytest.mark.parametrize("K,reps", [(1, 16), (16, 16), (17, 16), (32, 16)])
def test_policy_representatives_pair(bsa, K, reps):
    assert _policy(bsa, 1000, 1024, K, BF)["reps_per_lane"] == reps


@pytest.mark.parametrize("K,reps", [(65, 8), (96, 8)])
def test_policy_representatives_warp(bsa, K, reps):
    assert _policy(bsa, 1000, 1024, K, BF)["reps_per_lane"] == reps


@pytest.mark.parametrize("K", [33, 48, 64])
def test_policy_octet(bsa, K):
    """Octet path: 4 rows per warp, 4 warps per CTA, one item per warp; the
    overflow fallback's buffer fits in a warp's shared memory."""
    p = _policy(bsa, 10**6, 1024, K, BF)
    assert p["path"] == bsa.BSA_PATH_OCTET and p["reps_per_lane"] == 16
    assert p["grid"] == (10**6 // 4 + 3) // 4 and p["warps_per_cta"] == 4
    assert p["cand_capacity"] * 8 <= p["smem_bytes"] // p["warps_per_cta"]


def test_policy_split_only_for_few_long_rows(bsa):
    # 1024 bf16 tiles: group path, never split
    assert _policy(bsa, 8, 1024, 16, BF)["chunks_per_row"] == 1
    # 8192 tiles, few rows: split over up to 8 warps
    p = _policy(bsa, 48, 8192, 16, BF)
    assert p["path"] == bsa.BSA_PATH_SPLIT and p["chunks_per_row"] == 8
    # many rows fill the GPU by themselves
    assert _policy(bsa, 1 << 20, 8192, 16, BF)["chunks_per_row"] == 1
    # chunks shrink as rows grow
    assert _policy(bsa, 2432, 8192, 16, BF)["chunks_per_row"] == 2


def test_policy_long_rows(bsa):
    """Buffers wider than 2 KB (bf16 or fp32) with topk <= 64 and rows that
    are not split: the pair / octet path with long_rows, whose second launch
    (the wide path over the listed rows) has a persistent grid of 6 CTAs per
    SM and a workspace for the list; fewer rows are split over several
    warps, and 2 KB buffers and topk > 64 have no second launch."""
    for sms in (148, 152):
        for K, path, dt in ((16, bsa.BSA_PATH_PAIR, BF), (64, bsa.BSA_PATH_OCTET, BF),
                            (16, bsa.BSA_PATH_PAIR, FP)):
            for rows in (32 * sms, 16 * sms + 1, 10**6):
                p = _policy(bsa, rows, 8192, K, dt, sms)
                assert p["path"] == path and p["chunks_per_row"] == 1
                assert p["long_rows"] == 1 and p["long_grid"] == 6 * sms
            p = _policy(bsa, 16 * sms, 8192, K, dt, sms)
            assert p["path"] == bsa.BSA_PATH_SPLIT and p["chunks_per_row"] >= 2
            assert p["long_rows"] == 0 and p["long_grid"] == 0
    for M, dtype, K in ((1024, BF, 16), (1024, BF, 64), (512, FP, 16), (8192, BF, 65)):
        p = _policy(bsa, 10**6, M, K, dtype)
        assert p["long_rows"] == 0 and p["long_grid"] == 0
    # the list and its counter: 4 bytes per row, 256-byte aligned, plus 256
    rows = 10**6
    assert bsa.bsa_topk_workspace_bytes(rows // 2, 2, 8192, 16, BF) == \
        (rows * 4 + 255) // 256 * 256 + 256
    assert bsa.bsa_topk_workspace_bytes(rows // 2, 2, 1024, 16, BF) == 0


def test_policy_capacity_and_grid(bsa):
    p = _policy(bsa, 10**6, 1025, 65, BF)
    assert p["cand_capacity"] >= 65 + 32 * 8 and p["cand_capacity"] % 32 == 0
    assert p["smem_bytes"] == p["warps_per_cta"] * p["cand_capacity"] * 8
    assert p["grid"] == (10**6 + 7) // 8          # one row per warp, 8 warps per CTA
    g = _policy(bsa, 10**6, 1024, 16, BF)
    # pair path: one 16-row item per warp, 4 warps per CTA, no persistent cap
    assert g["path"] == bsa.BSA_PATH_PAIR and g["grid"] == (10**6 // 16 + 3) // 4
    # the overflow fallback's buffer fits in a pair warp's shared memory
    assert g["cand_capacity"] * 8 <= g["smem_bytes"] // g["warps_per_cta"]
    assert _policy(bsa, 10, 74, 16, BF)["grid"] == 1


def test_policy_rejects(bsa):
    L = bsa.lib()
    pol = bsa.LaunchPolicy()
    assert L.bsa_select_policy(10, 74, 16, 5, 152, ctypes.byref(pol)) == -4
    assert L.bsa_select_policy(10, 0, 1, 0, 152, ctypes.byref(pol)) == -2
    assert L.bsa_select_policy(10, 74, 75, 0, 152, ctypes.byref(pol)) == -3
    assert L.bsa_select_policy(10, 74, 16, 0, 152, None) == -1


def test_host_argument_checks_launch_nothing(bsa):
    """Invalid arguments are rejected on the host before any CUDA call."""
    L = bsa.lib()
    nul = ctypes.c_void_p(0)
    sel = L.bsa_topk_select
    tm = (4, 4)   # token-major output strides for H = 1, K = 4
    # K out of range, K < init + local, unknown dtype, bad sizes, null pointers
    assert sel(nul, 0, 4, 1, 32, 32, 32, nul, 0, 0, 0, nul, *tm, nul, 0, nul) == -3
    assert sel(nul, 0, 4, 1, 32, 32, 32, nul, 33, 0, 0, nul, *tm, nul, 0, nul) == -3
    assert sel(nul, 0, 4, 1, 32, 32, 32, nul, 2, 2, 1, nul, *tm, nul, 0, nul) == -3
    assert sel(nul, 9, 4, 1, 32, 32, 32, nul, 4, 1, 1, nul, *tm, nul, 0, nul) == -4
    assert sel(nul, 0, 4, 1, 0, 32, 32, nul, 4, 1, 1, nul, *tm, nul, 0, nul) == -2
    assert sel(nul, 0, 4, 2, 32, 40, 32, nul, 4, 1, 1, nul, *tm, nul, 0, nul) == -2
    assert sel(nul, 0, 4, 1, 32, 32, 32, nul, 4, 1, 1, nul, *tm, nul, 0, nul) == -1
    assert sel(ctypes.c_void_p(0x1001), 0, 4, 1, 32, 32, 32, ctypes.c_void_p(0x2000), 4, 1, 1,
               ctypes.c_void_p(0x3000), *tm, nul, 0, nul) == -7
    # empty batches are a no-op
    assert sel(nul, 0, 0, 1, 32, 32, 32, nul, 4, 1, 1, nul, *tm, nul, 0, nul) == 0
    tbl = L.bsa_build_sparse_block_table
    assert tbl(nul, 5, 1, 4, nul, 2, 3, nul, 2, nul, nul, nul) == -6
    assert tbl(nul, 4, 1, 0, nul, 2, 3, nul, 2, nul, nul, nul) == -3
    assert tbl(nul, 4, 1, 4, nul, 2, 3, nul, 2, nul, nul, nul) == -1
    fused = L.bsa_topk_select_sparse_table
    assert fused(nul, 0, 4, 0, 1, 32, 32, 32, nul, 4, 1, 1, nul, 3, nul, *tm, nul, nul, nul, 0,
                 nul) == -2
    assert fused(nul, 0, 4, 1, 1, 32, 32, 32, nul, 40, 1, 1, nul, 3, nul, *tm, nul, nul, nul, 0,
                 nul) == -3
    assert L.bsa_num_valid_pages_decode(nul, 4, 0, nul, nul) == -2
    assert L.bsa_num_valid_pages_decode(nul, 4, 1, nul, nul) == -1
    assert L.bsa_num_valid_pages_varlen(nul, nul, 2, -1, nul, nul) == -2


@pytest.mark.parametrize("T,H,K,ots,ohs,ok", [
    (5, 3, 4, 12, 4, True),      # token-major [T, H, K]
    (5, 3, 4, 4, 20, True),      # head-major [H, T, K] seen through transpose(0, 1)
    (5, 3, 4, 16, 4, True),      # padded token rows
    (5, 3, 4, 12, 3, False),     # slots of neighbouring heads overlap
    (5, 3, 4, 4, 19, False),     # the last token row of head 0 runs into head 1
    (5, 3, 4, 8, 4, False),      # token rows overlap the next token's heads
    (5, 1, 4, 4, 0, True),       # one head: its stride is irrelevant
    (1, 3, 4, 0, 4, True),       # one token: its stride is irrelevant
    (5, 1, 4, 3, 0, False),
    (5, 3, 4, -12, 4, False),
])
def test_output_layout_checks(bsa, T, H, K, ots, ohs, ok):
    """Output strides are checked on the host: any layout in which two rows
    (t, h) cannot overlap is accepted (the call then fails on its NULL
    pointers, -1); others are rejected (-2)."""
    L = bsa.lib()
    nul = ctypes.c_void_p(0)
    rc = L.bsa_topk_select(nul, 0, T, H, 32, 32 * H, 32, nul, K, 1, 1, nul, ots, ohs, nul, 0,
                           nul)
    assert rc == (-1 if ok else -2)
    rc = L.bsa_topk_select_sparse_table(nul, 0, T, 1, H, 32, 32 * H, 32, nul, K, 1, 1, nul, 3,
                                        ctypes.c_void_p(0x1000), ots, ohs, nul, nul, nul, 0, nul)
    assert rc == (-1 if ok else -2)


def test_binding_rejects_wrong_shapes_before_any_launch(bsa, monkeypatch):
    """The binding checks every tensor's shape, dtype and device before it
    calls the library; a mismatch is a ValueError, never an out-of-bounds
    device access.  The C entry points are replaced by a recorder, so a
    launch that should not happen is seen without a GPU."""
    import torch
    calls = []

    class FakeLib:
        def __getattr__(self, name):
            def rec(*a):
                calls.append(name)
                return 0
            return rec

    def meta(shape, dtype=torch.int32):
        return torch.empty(shape, dtype=dtype, device="meta")

    monkeypatch.setattr(bsa, "lib", lambda: FakeLib())
    # meta tensors (no memory) stand in for device tensors; is_cuda is
    # patched so that the binding's shape checks are the ones reached
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    T, H, K, M = 6, 2, 4, 40
    scores = meta((T, H, M), torch.bfloat16)
    good_nvp = meta((T,))
    with pytest.raises(ValueError, match="num_valid_pages"):
        bsa.bsa_topk_select(scores, meta((T + 1,)), K, out_idx=meta((T, H, K)))
    with pytest.raises(ValueError, match="out_idx"):
        bsa.bsa_topk_select(scores, good_nvp, K, out_idx=meta((T, H, K + 1)))
    with pytest.raises(ValueError, match="out_idx"):
        bsa.bsa_topk_select(scores, good_nvp, K, out_idx=meta((H, T, K)).transpose(1, 2)[:, :, :])
    seq = meta((3,))
    with pytest.raises(ValueError, match="block_table"):
        bsa.bsa_topk_select_sparse_table(scores, seq, 2, K, 1, 1, meta((4, 9)),
                                         out_idx=meta((T, H, K)), sparse_bt=meta((T, H, 8 * K)),
                                         sparse_ctx=meta((T, H)))
    with pytest.raises(ValueError, match="sparse_bt"):
        bsa.bsa_topk_select_sparse_table(scores, seq, 2, K, 1, 1, meta((3, 9)),
                                         out_idx=meta((T, H, K)), sparse_bt=meta((T, H, 8 * K - 1)),
                                         sparse_ctx=meta((T, H)))
    with pytest.raises(ValueError, match="sparse_ctx"):
        bsa.bsa_topk_select_sparse_table(scores, seq, 2, K, 1, 1, meta((3, 9)),
                                         out_idx=meta((T, H, K)), sparse_bt=meta((T, H, 8 * K)),
                                         sparse_ctx=meta((T,)))
    with pytest.raises(ValueError, match="sparse_bt"):
        bsa.bsa_build_sparse_block_table(meta((T, H, K)), meta((3, 9)), seq, 2,
                                         sparse_bt=meta((T, H, 8)), sparse_ctx=meta((T, H)))
    with pytest.raises(ValueError, match="block_table"):
        bsa.bsa_build_sparse_block_table(meta((T, H, K)), meta((2, 9)), seq, 2)
    with pytest.raises(ValueError, match="out"):
        bsa.bsa_num_valid_pages_decode(seq, 2, out=meta((5,)))
    with pytest.raises(ValueError, match="cu_seqlens_q"):
        bsa.bsa_num_valid_pages_varlen(meta((3,)), meta((3,)), 10)
    with pytest.raises(ValueError, match="out_idx"):
        bsa.bsa_topk_select_noalloc(scores, good_nvp, K, out_idx=meta((T, H, K - 1)))
    assert calls == [], calls
