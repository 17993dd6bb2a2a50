"""CPU oracle for the block-sparse attention top-k selection path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``block_sparse_attention_topk_gb300``) never imports it and shares no
code with it.

The arithmetic lives in ``bsa_oracle.c`` (plain single-threaded C, built here
with the host compiler on first use); this module only compiles it, loads it
with ctypes and marshals numpy arrays.  Every function cites, in the C
source, the passage of the vLLM PR reports it follows.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"libbsa_oracle_{platform.machine()}.so")

BF16 = 0
FP32 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build`` (host gcc, no GPU needed)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _declare(lib):
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64 = ctypes.c_int64
    i32 = ctypes.c_int32
    lib.oracle_total_order_cmp.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int]
    lib.oracle_total_order_cmp.restype = ctypes.c_int
    lib.oracle_num_valid_pages_decode.argtypes = [i32p, i64, i32, i32p]
    lib.oracle_num_valid_pages_varlen.argtypes = [i32p, i32p, i64, i32p]
    lib.oracle_topk_select.argtypes = [ctypes.c_void_p, ctypes.c_int, i64, i64, i64,
                                       i64, i64, i32p, i32, i32, i32, i32p]
    lib.oracle_build_sparse_block_table.argtypes = [i32p, i64, i64, i32, i32p, i64,
                                                    i64, i32p, i32, i32p, i32p]
    lib.oracle_topk_select_sparse_table.argtypes = [
        ctypes.c_void_p, ctypes.c_int, i64, i32, i64, i64, i64, i64, i32p, i32, i32,
        i32, i32p, i64, i32p, i32p, i32p]
    u16p = ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_index_scores.argtypes = [u16p, u16p, i64, i32p, i64, i32p, i64, i32, i64, i64,
                                        i64, ctypes.POINTER(ctypes.c_double)]
    lib.oracle_sparse_decode_attention.argtypes = [u16p, u16p, u16p, i64, i32p, i32p, i64, i64,
                                                   i64, i64, i32, ctypes.c_double,
                                                   ctypes.POINTER(ctypes.c_double)]
    for name in ("oracle_num_valid_pages_decode", "oracle_num_valid_pages_varlen",
                 "oracle_topk_select", "oracle_build_sparse_block_table",
                 "oracle_topk_select_sparse_table", "oracle_index_scores",
                 "oracle_sparse_decode_attention"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def load_library(path: str):
    """Load an oracle build from `path` (the mutant tests compile planted
    mistakes into a temporary copy and load it through this)."""
    return _declare(ctypes.CDLL(path))


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _score_bits(scores) -> tuple[np.ndarray, int]:
    """Accept a numpy uint16 (bf16 bits) / float32 / uint32 array or a CPU torch
    tensor of dtype bfloat16 / float32; return (contiguous bits array, dtype)."""
    if hasattr(scores, "detach"):  # torch tensor
        import torch
        t = scores.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return np.ascontiguousarray(t.view(torch.int16).numpy().view(np.uint16)), BF16
        if t.dtype == torch.float32:
            return np.ascontiguousarray(t.numpy().view(np.uint32)), FP32
        raise TypeError(f"unsupported score dtype {t.dtype}")
    a = np.asarray(scores)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    if a.dtype == np.float32:
        return np.ascontiguousarray(a.view(np.uint32)), FP32
    if a.dtype == np.uint32:
        return np.ascontiguousarray(a), FP32
    raise TypeError(f"unsupported score dtype {a.dtype}")


def total_order_cmp(a_bits: int, b_bits: int, dtype: int, lib=None) -> int:
    """IEEE 754 totalOrder of two bit patterns: -1, 0 or +1."""
    return int(_load(lib).oracle_total_order_cmp(a_bits & 0xFFFFFFFF, b_bits & 0xFFFFFFFF, dtype))


def num_valid_pages_decode(seq_lens, dql: int, lib=None) -> np.ndarray:
    s = _i32(seq_lens)
    out = np.zeros(s.shape[0] * dql, dtype=np.int32)
    rc = _load(lib).oracle_num_valid_pages_decode(_ptr(s), s.shape[0], dql, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_num_valid_pages_decode rc={rc}")
    return out


def num_valid_pages_varlen(cu_seqlens_q, prefix_lens, lib=None) -> np.ndarray:
    cu = _i32(cu_seqlens_q)
    pre = _i32(prefix_lens)
    out = np.zeros(int(cu[-1]), dtype=np.int32)
    rc = _load(lib).oracle_num_valid_pages_varlen(_ptr(cu), _ptr(pre), pre.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_num_valid_pages_varlen rc={rc}")
    return out


def topk_select(scores, nvp, K: int, num_init: int = 1, num_local: int = 1,
                token_stride: int | None = None, head_stride: int | None = None,
                T: int | None = None, H: int | None = None, M: int | None = None,
                lib=None) -> np.ndarray:
    """Top-k over a [T, H, M] score buffer (or a flat buffer with explicit
    strides); returns int32 [T, H, K]."""
    bits, dtype = _score_bits(scores)
    if T is None:
        T, H, M = bits.shape
    if head_stride is None:
        head_stride = M
    if token_stride is None:
        token_stride = H * M
    nv = _i32(nvp)
    assert nv.shape[0] == T
    out = np.full((T, H, K), -7, dtype=np.int32)
    rc = _load(lib).oracle_topk_select(bits.ctypes.data, dtype, T, H, M, token_stride,
                                    head_stride, _ptr(nv), K, num_init, num_local, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_topk_select rc={rc}")
    return out


def build_sparse_block_table(topk_idx, block_table, seq_lens, dql: int, lib=None):
    """Returns (sparse_bt int32 [T, H, K*8], sparse_ctx int32 [T, H])."""
    idx = _i32(topk_idx)
    T, H, K = idx.shape
    bt = _i32(block_table)
    B, MB = bt.shape
    s = _i32(seq_lens)
    sparse_bt = np.full((T, H, K * 8), -7, dtype=np.int32)
    sparse_ctx = np.full((T, H), -7, dtype=np.int32)
    rc = _load(lib).oracle_build_sparse_block_table(_ptr(idx), T, H, K, _ptr(bt), B, MB, _ptr(s),
                                                 dql, _ptr(sparse_bt), _ptr(sparse_ctx))
    if rc != 0:
        raise ValueError(f"oracle_build_sparse_block_table rc={rc}")
    return sparse_bt, sparse_ctx


def topk_select_sparse_table(scores, seq_lens, dql: int, K: int, num_init: int,
                             num_local: int, block_table, token_stride: int | None = None,
                             head_stride: int | None = None, H: int | None = None,
                             M: int | None = None, lib=None):
    """Returns (out_idx [T,H,K], sparse_bt [T,H,K*8], sparse_ctx [T,H]).
    `scores` is a [T, H, M] buffer, or a flat buffer with explicit H, M and
    strides (a capacity-wide or padded layout)."""
    bits, dtype = _score_bits(scores)
    if H is None:
        T, H, M = bits.shape
    s = _i32(seq_lens)
    B = s.shape[0]
    T = B * dql
    if bits.ndim == 3:
        assert bits.shape[0] == T
    bt = _i32(block_table)
    MB = bt.shape[1]
    if head_stride is None:
        head_stride = M
    if token_stride is None:
        token_stride = H * M
    out_idx = np.full((T, H, K), -7, dtype=np.int32)
    sparse_bt = np.full((T, H, K * 8), -7, dtype=np.int32)
    sparse_ctx = np.full((T, H), -7, dtype=np.int32)
    rc = _load(lib).oracle_topk_select_sparse_table(
        bits.ctypes.data, dtype, B, dql, H, M, token_stride, head_stride, _ptr(s), K,
        num_init, num_local, _ptr(bt), MB, _ptr(out_idx), _ptr(sparse_bt), _ptr(sparse_ctx))
    if rc != 0:
        raise ValueError(f"oracle_topk_select_sparse_table rc={rc}")
    return out_idx, sparse_bt, sparse_ctx


def _bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of a CPU torch bfloat16 tensor or a uint16 array."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype != torch.bfloat16:
            raise TypeError(f"expected bfloat16, got {t.dtype}")
        return np.ascontiguousarray(t.view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(np.asarray(x))
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bits, got {a.dtype}")
    return a


def index_scores(q, k, block_table, seq_lens, dql: int, M: int, lib=None) -> np.ndarray:
    """Index scores of decode rows in float64: q bf16 [T, H, D], k bf16
    [NB, D] (one pooled key per physical block), block_table int32 [B, MB],
    seq_lens int32 [B]; returns [T, H, M] (NaN past each row's causal
    count, -inf for causal blocks without a usable key)."""
    qb = _bf16_bits(q)
    kb = _bf16_bits(k)
    T, H, D = qb.shape
    NB = kb.shape[0]
    assert kb.shape[1] == D
    bt = _i32(block_table)
    B, MB = bt.shape
    s = _i32(seq_lens)
    assert s.shape[0] == B and T == B * dql
    out = np.empty((T, H, M), dtype=np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    rc = _load(lib).oracle_index_scores(qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), NB,
                                        _ptr(bt), MB, _ptr(s), B, dql, H, D, M,
                                        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError(f"oracle_index_scores rc={rc}")
    return out


def sparse_decode_attention(q, k_cache, v_cache, sparse_bt, sparse_ctx, scale: float,
                            lib=None) -> np.ndarray:
    """Sparse decode attention in float64: q bf16 [T, H, G, D], k_cache and
    v_cache bf16 [num_pages, 16, H, D], sparse_bt int32 [T, H, K*8],
    sparse_ctx int32 [T, H]; returns [T, H, G, D]."""
    qb = _bf16_bits(q)
    kb = _bf16_bits(k_cache)
    vb = _bf16_bits(v_cache)
    T, H, G, D = qb.shape
    NP = kb.shape[0]
    assert kb.shape == (NP, 16, H, D) and vb.shape == kb.shape
    bt = _i32(sparse_bt)
    ctx = _i32(sparse_ctx)
    assert bt.shape[:2] == (T, H) and bt.shape[2] % 8 == 0 and ctx.shape == (T, H)
    K = bt.shape[2] // 8
    out = np.empty((T, H, G, D), dtype=np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    rc = _load(lib).oracle_sparse_decode_attention(
        qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p), NP, _ptr(bt),
        _ptr(ctx), T, H, G, D, K, float(scale), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError(f"oracle_sparse_decode_attention rc={rc}")
    return out
