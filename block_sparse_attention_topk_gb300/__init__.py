"""GB300 (sm_103a) block-sparse attention top-k selection.

A thin Python binding over the C ABI in ``include/bsa_topk.h``: each
function here has the name of the C entry point it calls and only marshals
arguments (tensor pointers, strides, the current CUDA stream).  Every step of
the computation runs in the library's own CUDA kernels; there is no CPU or
PyTorch fallback -- importing this package fails if the library has not been
built (``python -m block_sparse_attention_topk_gb300.build``).

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

BSA_OK = 0
BSA_DTYPE_BF16 = 0
BSA_DTYPE_FP32 = 1
BSA_PATH_ROW = 0
BSA_PATH_SPLIT = 1
BSA_PATH_GROUP = 2
BSA_PATH_PAIR = 3
BSA_PATH_OCTET = 4
BSA_PATH_WIDE = 5
PAGE_SIZE = 128
PAGES_PER_SPARSE_BLOCK = 8
MAX_TOPK = 1024
MAX_K_TILES = 65536

_ERRORS = {-1: "BSA_ERR_NULL", -2: "BSA_ERR_SHAPE", -3: "BSA_ERR_TOPK", -4: "BSA_ERR_DTYPE",
           -5: "BSA_ERR_WORKSPACE", -6: "BSA_ERR_ROWS", -7: "BSA_ERR_ALIGN",
           -8: "BSA_ERR_CAPACITY"}
NOALLOC_SCRATCH_BYTES = 16 << 20

# Names of every extern "C" symbol the header declares (checked by the tests).
EXPORTED = [
    "bsa_status_string", "bsa_num_valid_pages_decode", "bsa_num_valid_pages_varlen",
    "bsa_topk_workspace_bytes", "bsa_topk_select", "bsa_build_sparse_block_table",
    "bsa_topk_select_sparse_table", "bsa_select_policy", "bsa_topk_select_noalloc",
    "bsa_index_score_topk_select", "bsa_sparse_decode_attention", "bsa_set_status_word",
    "bsa_read_status",
]
# bits of the device status word (bsa_set_status_word)
BSA_STATUS_BAD_BLOCK_ID = 0x1
BSA_STATUS_BAD_PAGE = 0x2
BSA_STATUS_BAD_CONTEXT = 0x4
MAX_ATTN_GROUP = 8
MAX_INDEX_DIM = 1024
MAX_INDEX_QUERIES = 16


class BsaError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        self.status = status
        name = _ERRORS.get(status, f"cudaError {status}" if status > 0 else str(status))
        super().__init__(f"{fn} failed: {name}: {message}")


class LaunchPolicy(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("vecs_per_lane", ctypes.c_int32),
                ("chunks_per_row", ctypes.c_int32), ("reps_per_lane", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("cand_capacity", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("long_rows", ctypes.c_int32), ("long_grid", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with "
                    "`python -m block_sparse_attention_topk_gb300.build`")
            L = ctypes.CDLL(path)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
            L.bsa_status_string.argtypes = [ctypes.c_int]
            L.bsa_status_string.restype = ctypes.c_char_p
            L.bsa_num_valid_pages_decode.argtypes = [vp, i64, i32, vp, vp]
            L.bsa_num_valid_pages_varlen.argtypes = [vp, vp, i64, i64, vp, vp]
            L.bsa_topk_workspace_bytes.argtypes = [i64, i64, i64, i32, i32]
            L.bsa_topk_workspace_bytes.restype = sz
            L.bsa_topk_select.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, i32, i32, i32,
                                          vp, i64, i64, vp, sz, vp]
            L.bsa_build_sparse_block_table.argtypes = [vp, i64, i64, i32, vp, i64, i64, vp, i32,
                                                       vp, vp, vp]
            L.bsa_topk_select_sparse_table.argtypes = [vp, i32, i64, i32, i64, i64, i64, i64, vp,
                                                       i32, i32, i32, vp, i64, vp, i64, i64, vp,
                                                       vp, vp, sz, vp]
            L.bsa_select_policy.argtypes = [i64, i64, i32, i32, i32, ctypes.POINTER(LaunchPolicy)]
            L.bsa_topk_select_noalloc.argtypes = [vp, i32, i64, i64, i64, i64, i64, vp, i32, i32,
                                                  i32, vp, vp]
            L.bsa_index_score_topk_select.argtypes = [vp, vp, i64, i64, i64, vp, i64, vp, i64,
                                                      i32, vp, i64, i64, i64, i32, i32, i32, vp,
                                                      i64, i64, vp, vp, vp]
            L.bsa_sparse_decode_attention.argtypes = [vp, vp, vp, i64, vp, vp, i64, i64, i64, i64,
                                                      i32, ctypes.c_float, vp, vp]
            L.bsa_set_status_word.argtypes = [vp]
            L.bsa_read_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, vp]
            for name in EXPORTED[1:]:
                if name != "bsa_topk_workspace_bytes":
                    getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != BSA_OK:
        raise BsaError(fn, status, lib().bsa_status_string(status).decode())


def _call(fn: str, device: torch.device, *args):
    """Calls C entry point `fn` with `device` current: the library takes the
    launch policy's SM count, the workspace size and its scratch address from
    the current device."""
    with torch.cuda.device(device):
        _check(fn, getattr(lib(), fn)(*args))


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dev_i32(t: torch.Tensor, name: str, device: torch.device | None = None,
             shape: tuple | None = None) -> torch.Tensor:
    """A contiguous int32 CUDA tensor, on `device` and of `shape` when given;
    raises ValueError before anything is launched otherwise."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32 \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _out_idx(t: torch.Tensor, T: int, H: int, K: int, device: torch.device):
    """An int32 [T, H, K] output view whose K slots are contiguous (token-major,
    or a transpose(0, 1) view of a head-major [H, T, K] buffer); returns its
    (token, head) element strides."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32:
        raise ValueError("out_idx must be an int32 CUDA tensor")
    if t.device != device:
        raise ValueError(f"out_idx is on {t.device}, expected {device}")
    if tuple(t.shape) != (T, H, K):
        raise ValueError(f"out_idx has shape {tuple(t.shape)}, expected {(T, H, K)}")
    if K > 1 and t.stride(2) != 1:
        raise ValueError("out_idx must be contiguous along its topk dimension")
    return t.stride(0), t.stride(1)


def _score_dtype(scores: torch.Tensor) -> int:
    if scores.dtype == torch.bfloat16:
        return BSA_DTYPE_BF16
    if scores.dtype == torch.float32:
        return BSA_DTYPE_FP32
    raise ValueError(f"scores must be bfloat16 or float32, not {scores.dtype}")


# One workspace per (device, stream), grown on demand (the library clears the
# parts it needs cleared on every call).  Calls on one stream run in order,
# so they may share it; calls on different streams get different buffers.
_ws_cache: dict = {}
_ws_lock = threading.Lock()


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    key = (device.type, device.index, torch.cuda.current_stream(device).cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def _workspace_arg(workspace: torch.Tensor | None, device: torch.device, need: int):
    if workspace is None:
        workspace = _workspace(device, need)
    elif not workspace.is_cuda or workspace.device != device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return workspace, nbytes


def bsa_topk_workspace_bytes(T: int, H: int, M: int, K: int, dtype: int,
                             device: torch.device | None = None) -> int:
    """Workspace bytes for these sizes on `device` (default: the current one)."""
    if device is None:
        return int(lib().bsa_topk_workspace_bytes(T, H, M, K, dtype))
    with torch.cuda.device(device):
        return int(lib().bsa_topk_workspace_bytes(T, H, M, K, dtype))


def bsa_select_policy(rows: int, M: int, K: int, dtype: int, num_sms: int = 152) -> dict:
    pol = LaunchPolicy()
    _check("bsa_select_policy",
           lib().bsa_select_policy(rows, M, K, dtype, num_sms, ctypes.byref(pol)))
    return pol.as_dict()


def bsa_num_valid_pages_decode(seq_lens: torch.Tensor, decode_query_len: int,
                               out: torch.Tensor | None = None) -> torch.Tensor:
    dev = seq_lens.device
    _dev_i32(seq_lens, "seq_lens")
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be 1-D [num_reqs]")
    T = seq_lens.shape[0] * decode_query_len
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=dev)
    _dev_i32(out, "out", dev, (T,))
    _call("bsa_num_valid_pages_decode", dev, _ptr(seq_lens), seq_lens.shape[0],
          decode_query_len, _ptr(out), _stream(dev))
    return out


def bsa_num_valid_pages_varlen(cu_seqlens_q: torch.Tensor, prefix_lens: torch.Tensor,
                               total_q: int, out: torch.Tensor | None = None) -> torch.Tensor:
    dev = cu_seqlens_q.device
    _dev_i32(prefix_lens, "prefix_lens", dev)
    if prefix_lens.dim() != 1:
        raise ValueError("prefix_lens must be 1-D [num_seqs]")
    _dev_i32(cu_seqlens_q, "cu_seqlens_q", dev, (prefix_lens.shape[0] + 1,))
    if out is None:
        out = torch.empty(total_q, dtype=torch.int32, device=dev)
    _dev_i32(out, "out", dev, (total_q,))
    _call("bsa_num_valid_pages_varlen", dev, _ptr(cu_seqlens_q), _ptr(prefix_lens),
          prefix_lens.shape[0], total_q, _ptr(out), _stream(dev))
    return out


def _score_view(scores: torch.Tensor, M: int | None):
    if not isinstance(scores, torch.Tensor) or scores.dim() != 3 or not scores.is_cuda:
        raise ValueError("scores must be a 3-D CUDA tensor [T, H, tiles]")
    if scores.shape[2] > 1 and scores.stride(2) != 1:
        raise ValueError("scores must be contiguous along the tile dimension")
    T, H, cap = scores.shape
    M = cap if M is None else int(M)
    if M > cap:
        raise ValueError(f"M={M} exceeds the tile dimension {cap}")
    return T, H, M, scores.stride(0), scores.stride(1)


def bsa_topk_select(scores: torch.Tensor, num_valid_pages: torch.Tensor, K: int,
                    num_init: int = 1, num_local: int = 1, out_idx: torch.Tensor | None = None,
                    M: int | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """scores [T, H, tiles] (bf16/fp32, tile dim contiguous; M = tiles used,
    default all), num_valid_pages int32[T] -> out_idx int32 [T, H, K].  A
    given out_idx may be any [T, H, K] view with contiguous topk slots, e.g.
    ``buf.transpose(0, 1)`` of a head-major [H, T, K] buffer."""
    T, H, M, ts, hs = _score_view(scores, M)
    dt = _score_dtype(scores)
    dev = scores.device
    _dev_i32(num_valid_pages, "num_valid_pages", dev, (T,))
    if out_idx is None:
        out_idx = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    ots, ohs = _out_idx(out_idx, T, H, K, dev)
    need = bsa_topk_workspace_bytes(T, H, M, K, dt, dev)
    workspace, wbytes = _workspace_arg(workspace, dev, need)
    _call("bsa_topk_select", dev, _ptr(scores), dt, T, H, M, ts, hs, _ptr(num_valid_pages), K,
          num_init, num_local, _ptr(out_idx), ots, ohs, _ptr(workspace), wbytes, _stream(dev))
    return out_idx


def bsa_build_sparse_block_table(topk_idx: torch.Tensor, block_table: torch.Tensor,
                                 seq_lens: torch.Tensor, decode_query_len: int,
                                 sparse_bt: torch.Tensor | None = None,
                                 sparse_ctx: torch.Tensor | None = None):
    """topk_idx int32 [T, H, K] -> (sparse_bt int32 [T, H, K*8], sparse_ctx int32 [T, H])."""
    dev = topk_idx.device
    _dev_i32(topk_idx, "topk_idx")
    if topk_idx.dim() != 3:
        raise ValueError("topk_idx must be [T, H, K]")
    T, H, K = topk_idx.shape
    _dev_i32(seq_lens, "seq_lens", dev)
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be 1-D [num_reqs]")
    B = seq_lens.shape[0]
    _dev_i32(block_table, "block_table", dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table has shape {tuple(block_table.shape)}, expected "
                         f"[{B}, max_blocks]")
    MB = block_table.shape[1]
    if sparse_bt is None:
        sparse_bt = torch.empty((T, H, K * PAGES_PER_SPARSE_BLOCK), dtype=torch.int32, device=dev)
    _dev_i32(sparse_bt, "sparse_bt", dev, (T, H, K * PAGES_PER_SPARSE_BLOCK))
    if sparse_ctx is None:
        sparse_ctx = torch.empty((T, H), dtype=torch.int32, device=dev)
    _dev_i32(sparse_ctx, "sparse_ctx", dev, (T, H))
    _call("bsa_build_sparse_block_table", dev, _ptr(topk_idx), T, H, K, _ptr(block_table), B,
          MB, _ptr(seq_lens), decode_query_len, _ptr(sparse_bt), _ptr(sparse_ctx), _stream(dev))
    return sparse_bt, sparse_ctx


def bsa_topk_select_sparse_table(scores: torch.Tensor, seq_lens: torch.Tensor,
                                 decode_query_len: int, K: int, num_init: int, num_local: int,
                                 block_table: torch.Tensor, want_idx: bool = True,
                                 out_idx: torch.Tensor | None = None,
                                 sparse_bt: torch.Tensor | None = None,
                                 sparse_ctx: torch.Tensor | None = None, M: int | None = None,
                                 workspace: torch.Tensor | None = None):
    """Fused decode select + sparse table over the first num_reqs *
    decode_query_len token rows of `scores`.  Returns (out_idx or None,
    sparse_bt, sparse_ctx); out_idx may be a strided view as for
    bsa_topk_select."""
    _, H, M, ts, hs = _score_view(scores, M)
    dt = _score_dtype(scores)
    dev = scores.device
    _dev_i32(seq_lens, "seq_lens", dev)
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be 1-D [num_reqs]")
    B = seq_lens.shape[0]
    _dev_i32(block_table, "block_table", dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table has shape {tuple(block_table.shape)}, expected "
                         f"[{B}, max_blocks]")
    MB = block_table.shape[1]
    T = B * decode_query_len
    if scores.shape[0] < T:
        raise ValueError(f"scores holds {scores.shape[0]} token rows, need {T}")
    if want_idx and out_idx is None:
        out_idx = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    ots, ohs = (H * K, K) if out_idx is None else _out_idx(out_idx, T, H, K, dev)
    if sparse_bt is None:
        sparse_bt = torch.empty((T, H, K * PAGES_PER_SPARSE_BLOCK), dtype=torch.int32, device=dev)
    _dev_i32(sparse_bt, "sparse_bt", dev, (T, H, K * PAGES_PER_SPARSE_BLOCK))
    if sparse_ctx is None:
        sparse_ctx = torch.empty((T, H), dtype=torch.int32, device=dev)
    _dev_i32(sparse_ctx, "sparse_ctx", dev, (T, H))
    need = bsa_topk_workspace_bytes(T, H, M, K, dt, dev)
    workspace, wbytes = _workspace_arg(workspace, dev, need)
    _call("bsa_topk_select_sparse_table", dev, _ptr(scores), dt, B, decode_query_len, H, M, ts,
          hs, _ptr(seq_lens), K, num_init, num_local, _ptr(block_table), MB, _ptr(out_idx), ots,
          ohs, _ptr(sparse_bt), _ptr(sparse_ctx), _ptr(workspace), wbytes, _stream(dev))
    return out_idx, sparse_bt, sparse_ctx


def bsa_topk_select_noalloc(scores: torch.Tensor, num_valid_pages: torch.Tensor, K: int,
                            num_init: int = 1, num_local: int = 1,
                            out_idx: torch.Tensor | None = None,
                            M: int | None = None) -> torch.Tensor:
    """bsa_topk_select without a workspace argument, for callers that cannot
    allocate device memory: the library's own fixed device array serves as
    scratch (see include/bsa_topk.h).  Same results as bsa_topk_select;
    out_idx is token-major and contiguous."""
    T, H, M, ts, hs = _score_view(scores, M)
    dt = _score_dtype(scores)
    dev = scores.device
    _dev_i32(num_valid_pages, "num_valid_pages", dev, (T,))
    if out_idx is None:
        out_idx = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    _dev_i32(out_idx, "out_idx", dev, (T, H, K))
    _call("bsa_topk_select_noalloc", dev, _ptr(scores), dt, T, H, M, ts, hs,
          _ptr(num_valid_pages), K, num_init, num_local, _ptr(out_idx), _stream(dev))
    return out_idx


def bsa_index_score_topk_select(q_idx: torch.Tensor, k_idx: torch.Tensor,
                                block_table: torch.Tensor, seq_lens: torch.Tensor,
                                decode_query_len: int, K: int, num_init: int = 1,
                                num_local: int = 1, M: int | None = None,
                                scores: torch.Tensor | None = None,
                                out_idx: torch.Tensor | None = None, with_table: bool = False,
                                sparse_bt: torch.Tensor | None = None,
                                sparse_ctx: torch.Tensor | None = None):
    """Fused index score + select of decode rows.  q_idx bf16 [T, H, D],
    k_idx bf16 [num_phys_blocks, D] (one pooled key per physical block),
    block_table int32 [num_reqs, max_blocks], seq_lens int32 [num_reqs].
    `scores` is the fp32 unified buffer [T, H, tiles] (tile dim contiguous;
    M = tiles used, default all); by default a new one pre-filled with -inf.
    Returns (scores, out_idx, sparse_bt or None, sparse_ctx or None)."""
    dev = q_idx.device
    if not isinstance(q_idx, torch.Tensor) or not q_idx.is_cuda or q_idx.dim() != 3 \
            or q_idx.dtype != torch.bfloat16 or not q_idx.is_contiguous():
        raise ValueError("q_idx must be a contiguous bf16 CUDA tensor [T, H, D]")
    T, H, D = q_idx.shape
    if not isinstance(k_idx, torch.Tensor) or k_idx.device != dev or k_idx.dim() != 2 \
            or k_idx.dtype != torch.bfloat16 or not k_idx.is_contiguous() or k_idx.shape[1] != D:
        raise ValueError(f"k_idx must be a contiguous bf16 tensor [num_phys_blocks, {D}] on {dev}")
    _dev_i32(seq_lens, "seq_lens", dev)
    if seq_lens.dim() != 1:
        raise ValueError("seq_lens must be 1-D [num_reqs]")
    B = seq_lens.shape[0]
    if T != B * decode_query_len:
        raise ValueError(f"q_idx holds {T} token rows, expected {B} x {decode_query_len}")
    _dev_i32(block_table, "block_table", dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError(f"block_table has shape {tuple(block_table.shape)}, expected "
                         f"[{B}, max_blocks]")
    MB = block_table.shape[1]
    if scores is None:
        cap = MB if M is None else int(M)
        scores = torch.full((T, H, cap), float("-inf"), dtype=torch.float32, device=dev)
    if scores.dtype != torch.float32 or scores.device != dev or scores.dim() != 3 \
            or tuple(scores.shape[:2]) != (T, H):
        raise ValueError(f"scores must be an fp32 tensor [{T}, {H}, tiles] on {dev}")
    _, _, M, ts, hs = _score_view(scores, M)
    if out_idx is None:
        out_idx = torch.empty((T, H, K), dtype=torch.int32, device=dev)
    ots, ohs = _out_idx(out_idx, T, H, K, dev)
    if with_table or sparse_bt is not None or sparse_ctx is not None:
        if sparse_bt is None:
            sparse_bt = torch.empty((T, H, K * PAGES_PER_SPARSE_BLOCK), dtype=torch.int32,
                                    device=dev)
        _dev_i32(sparse_bt, "sparse_bt", dev, (T, H, K * PAGES_PER_SPARSE_BLOCK))
        if sparse_ctx is None:
            sparse_ctx = torch.empty((T, H), dtype=torch.int32, device=dev)
        _dev_i32(sparse_ctx, "sparse_ctx", dev, (T, H))
    _call("bsa_index_score_topk_select", dev, _ptr(q_idx), _ptr(k_idx), k_idx.shape[0], H, D,
          _ptr(block_table), MB, _ptr(seq_lens), B, decode_query_len, _ptr(scores), M, ts, hs, K,
          num_init, num_local, _ptr(out_idx), ots, ohs, _ptr(sparse_bt), _ptr(sparse_ctx),
          _stream(dev))
    return scores, out_idx, sparse_bt, sparse_ctx


def bsa_sparse_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                sparse_bt: torch.Tensor, sparse_ctx: torch.Tensor,
                                scale: float | None = None,
                                out: torch.Tensor | None = None) -> torch.Tensor:
    """Sparse decode attention over the page-16 table.  q bf16 [T, H, G, D],
    k_cache / v_cache bf16 [num_pages, 16, H, D], sparse_bt int32
    [T, H, K*8], sparse_ctx int32 [T, H]; returns fp32 [T, H, G, D].  The
    scale defaults to 1 / sqrt(D)."""
    dev = q.device
    if not isinstance(q, torch.Tensor) or not q.is_cuda or q.dim() != 4 \
            or q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 CUDA tensor [T, H, G, D]")
    T, H, G, D = q.shape
    for name, c in (("k_cache", k_cache), ("v_cache", v_cache)):
        if not isinstance(c, torch.Tensor) or c.device != dev or c.dtype != torch.bfloat16 \
                or not c.is_contiguous() or c.dim() != 4 or tuple(c.shape[1:]) != (16, H, D):
            raise ValueError(f"{name} must be a contiguous bf16 tensor [num_pages, 16, {H}, {D}] "
                             f"on {dev}")
    if k_cache.shape[0] != v_cache.shape[0]:
        raise ValueError("k_cache and v_cache hold different page counts")
    _dev_i32(sparse_bt, "sparse_bt", dev)
    if sparse_bt.dim() != 3 or tuple(sparse_bt.shape[:2]) != (T, H) or sparse_bt.shape[2] % 8:
        raise ValueError(f"sparse_bt must be [{T}, {H}, K*8]")
    K = sparse_bt.shape[2] // PAGES_PER_SPARSE_BLOCK
    _dev_i32(sparse_ctx, "sparse_ctx", dev, (T, H))
    if out is None:
        out = torch.empty((T, H, G, D), dtype=torch.float32, device=dev)
    if out.dtype != torch.float32 or out.device != dev or not out.is_contiguous() \
            or tuple(out.shape) != (T, H, G, D):
        raise ValueError(f"out must be a contiguous fp32 tensor [{T}, {H}, {G}, {D}] on {dev}")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    _call("bsa_sparse_decode_attention", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache),
          k_cache.shape[0], _ptr(sparse_bt), _ptr(sparse_ctx), T, H, G, D, K, ctypes.c_float(scale),
          _ptr(out), _stream(dev))
    return out


_status_words: dict[int, torch.Tensor] = {}


def bsa_set_status_word(word: torch.Tensor | None, device: torch.device | None = None) -> None:
    """Registers `word`, a one-element int32 CUDA tensor that the caller has
    zeroed, as the status word of its device, or with None unregisters the
    word of `device` (default: the current device).  The kernels of later
    calls on that device set BSA_STATUS_* bits in it instead of faulting on
    invalid block-table entries, pages or context lengths.  The binding keeps
    a reference to the tensor while it is registered."""
    if word is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        _call("bsa_set_status_word", dev, ctypes.c_void_p(0))
        _status_words.pop(dev.index, None)
        return
    if not isinstance(word, torch.Tensor) or not word.is_cuda or word.dtype != torch.int32 \
            or word.numel() != 1:
        raise ValueError("word must be a one-element int32 CUDA tensor")
    _call("bsa_set_status_word", word.device, _ptr(word))
    _status_words[word.device.index] = word


def bsa_read_status(clear: bool = True, device: torch.device | None = None) -> int:
    """The status word of `device` (default: the current device) once the work
    queued so far on its current stream is done, cleared when `clear`; 0 when
    no word is registered."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    out = ctypes.c_uint32(0)
    _call("bsa_read_status", dev, ctypes.byref(out), int(bool(clear)), _stream(dev))
    return int(out.value)
