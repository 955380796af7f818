"""GB300 (sm_103a) DeepSeek-V4 sparse-MLA decode: Python binding of the C ABI (include/dsv4.h).

The functions below carry the C entry points' names and only marshal
arguments: they take torch tensors that already live on the GPU, read their
pointers, sizes and strides, and call libdsv4_gb300.so through ctypes on the
current torch stream.  Every step of the decode runs in the library's CUDA
kernels; there is no Python or CPU fallback, and importing this package
raises if the library has not been built (``sparse_mla_decode_combine_gb300.build.build()``).

Status codes are returned as ints (``DSV4_OK`` == 0); ``check()`` turns a
non-zero code into an exception.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

DSV4_OK = 0
DSV4_ERR_INVALID_ARG = 1
DSV4_ERR_BAD_INDEX = 2
DSV4_ERR_TIMEOUT = 3
DSV4_ERR_CUDA = 4
DSV4_ERR_UNSUPPORTED = 5
STATUS_NAMES = {0: "DSV4_OK", 1: "DSV4_ERR_INVALID_ARG", 2: "DSV4_ERR_BAD_INDEX", 3: "DSV4_ERR_TIMEOUT",
                4: "DSV4_ERR_CUDA", 5: "DSV4_ERR_UNSUPPORTED"}

EXPORTED = ("dsv4_combine_topk_swa_indices", "dsv4_combine_topk_swa_indices_compressed", "dsv4_topk_select",
            "dsv4_qnorm_rope_kv_insert", "dsv4_selftest_wait_timeout",
            "dsv4_sparse_mla_decode_workspace_size", "dsv4_sparse_mla_decode", "dsv4_sparse_mla_decode_trace",
            "dsv4_sparse_mla_decode_noalloc", "dsv4_sparse_mla_decode_mtp_union",
            "dsv4_sparse_mla_decode_mtp_union_workspace_size", "dsv4_get_device_status")


class Dsv4Error(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}" if what else STATUS_NAMES.get(code, str(code)))
        self.code = code


def check(code: int, what: str = "") -> None:
    if code != DSV4_OK:
        raise Dsv4Error(code, what)


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load libdsv4_gb300.so (raises FileNotFoundError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise FileNotFoundError(f"CUDA library not built: {path} (run sparse_mla_decode_combine_gb300.build.build())")
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.dsv4_combine_topk_swa_indices.restype = ctypes.c_int
    lib.dsv4_combine_topk_swa_indices.argtypes = [P, i64, i32, P, P, i32, i32, P, i64, i32, P, P]
    lib.dsv4_combine_topk_swa_indices_compressed.restype = ctypes.c_int
    lib.dsv4_combine_topk_swa_indices_compressed.argtypes = [P, i64, i32, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                             P, i64, i32, P, P]
    lib.dsv4_selftest_wait_timeout.restype = ctypes.c_int
    lib.dsv4_selftest_wait_timeout.argtypes = [i64, P]
    lib.dsv4_qnorm_rope_kv_insert.restype = ctypes.c_int
    lib.dsv4_qnorm_rope_kv_insert.argtypes = [P, i64, P, i64, i32, i32, P, ctypes.c_float, P, i64, P, P, P, i32, P,
                                              i64, P]
    lib.dsv4_topk_select.restype = ctypes.c_int
    lib.dsv4_topk_select.argtypes = [P, i64, i32, P, i32, i32, P, i64, P, P]
    lib.dsv4_sparse_mla_decode_workspace_size.restype = ctypes.c_size_t
    lib.dsv4_sparse_mla_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.dsv4_sparse_mla_decode.restype = ctypes.c_int
    lib.dsv4_sparse_mla_decode.argtypes = [P, i64, P, i32, i32, P, i64, i32, i32, P, P, i64, i32, P, P, i32, i32,
                                           i32, P, ctypes.c_float, P, P, P, ctypes.c_size_t, P]
    lib.dsv4_sparse_mla_decode_trace.restype = ctypes.c_int
    lib.dsv4_sparse_mla_decode_trace.argtypes = [P, i64, P, i32, i32, P, i64, i32, i32, P, P, i64, i32, P, P, i32, i32,
                                                 i32, P, ctypes.c_float, P, P, P, ctypes.c_size_t, P, i64, i32, P, P]
    lib.dsv4_sparse_mla_decode_noalloc.restype = ctypes.c_int
    lib.dsv4_sparse_mla_decode_noalloc.argtypes = [P, i64, P, i32, i32, P, i64, i32, i32, P, P, i64, i32, P, P, i32,
                                                   i32, i32, P, ctypes.c_float, P, P, P]
    lib.dsv4_sparse_mla_decode_mtp_union.restype = ctypes.c_int
    lib.dsv4_sparse_mla_decode_mtp_union.argtypes = [P, i64, P, i32, i32, P, i64, i32, i32, P, P, i64, i32, P, P, i32,
                                                     i32, i32, P, ctypes.c_float, P, P, P, ctypes.c_size_t, P]
    lib.dsv4_sparse_mla_decode_mtp_union_workspace_size.restype = ctypes.c_size_t
    lib.dsv4_sparse_mla_decode_mtp_union_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.dsv4_get_device_status.restype = ctypes.c_int
    lib.dsv4_get_device_status.argtypes = [P]
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: Optional[torch.Tensor], dtype, name: str, ndim: Optional[int] = None):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {t.dim()}")
    if t.numel() > 0 and t.dim() > 0 and t.stride(-1) != 1:
        raise ValueError(f"{name}: last dim must be contiguous")


def dsv4_combine_topk_swa_indices(topk_idx: torch.Tensor, topk_lens: Optional[torch.Tensor], seq_lens: torch.Tensor,
                                  window: int, combined: torch.Tensor, combined_lens: torch.Tensor,
                                  stream=None) -> int:
    """topk_idx int32 [T, K]; topk_lens int32 [T] or None; seq_lens int32 [T];
    combined int32 [T, C] (C >= K + window); combined_lens int32 [T]."""
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(combined, torch.int32, "combined", 2)
    _need(combined_lens, torch.int32, "combined_lens", 1)
    T, K = topk_idx.shape
    return load_library().dsv4_combine_topk_swa_indices(
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(topk_lens), _ptr(seq_lens), T,
        int(window), _ptr(combined), max(combined.stride(0), combined.shape[1]), combined.shape[1],
        _ptr(combined_lens), _stream(stream))


def dsv4_combine_topk_swa_indices_compressed(topk_idx: torch.Tensor, query_start_loc: torch.Tensor,
                                             seq_lens: torch.Tensor, gather_lens: torch.Tensor, region_stride: int,
                                             compressed_len: int, top_k: int, compress_ratio: int, window: int,
                                             combined: torch.Tensor, combined_lens: torch.Tensor, stream=None) -> int:
    """topk_idx int32 [T, K]; query_start_loc int32 [R + 1]; seq_lens, gather_lens int32 [R];
    combined int32 [T, C] (C >= top_k + window); combined_lens int32 [T]."""
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(gather_lens, torch.int32, "gather_lens", 1)
    _need(combined, torch.int32, "combined", 2)
    _need(combined_lens, torch.int32, "combined_lens", 1)
    T, K = topk_idx.shape
    return load_library().dsv4_combine_topk_swa_indices_compressed(
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(query_start_loc), _ptr(seq_lens),
        _ptr(gather_lens), query_start_loc.numel() - 1, T, int(region_stride), int(compressed_len), int(top_k),
        int(compress_ratio), int(window), _ptr(combined), max(combined.stride(0), combined.shape[1]),
        combined.shape[1], _ptr(combined_lens), _stream(stream))


def dsv4_selftest_wait_timeout(cycles: int, stream=None) -> int:
    """One bounded wait on an mbarrier nothing arrives on (see include/dsv4.h)."""
    return load_library().dsv4_selftest_wait_timeout(int(cycles), _stream(stream))


def dsv4_qnorm_rope_kv_insert(q: torch.Tensor, q_out: torch.Tensor, kv: torch.Tensor, positions: torch.Tensor,
                              slot_mapping: torch.Tensor, cos_sin_cache: torch.Tensor, kv_cache: torch.Tensor,
                              q_norm_weight: Optional[torch.Tensor] = None, eps: float = 1e-6, stream=None) -> int:
    """q, q_out bf16 [T, H, 576] (heads contiguous); kv bf16 [T, 576]; positions, slot_mapping int64 [T];
    cos_sin_cache float32 [max_position, 64]; kv_cache uint8 [..., 656] (slots in order);
    q_norm_weight float32 [576] or None."""
    _need(q, torch.bfloat16, "q", 3)
    _need(q_out, torch.bfloat16, "q_out", 3)
    _need(kv, torch.bfloat16, "kv", 2)
    _need(positions, torch.int64, "positions", 1)
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    _need(cos_sin_cache, torch.float32, "cos_sin_cache", 2)
    _need(kv_cache, torch.uint8, "kv_cache")
    _need(q_norm_weight, torch.float32, "q_norm_weight", 1)
    T, H, _ = q.shape
    if q.stride(1) != 576 or q_out.stride(1) != 576:
        raise ValueError("q, q_out: heads must be contiguous")
    if not kv_cache.is_contiguous():
        raise ValueError("kv_cache: must be contiguous")
    return load_library().dsv4_qnorm_rope_kv_insert(
        _ptr(q), q.stride(0), _ptr(q_out), q_out.stride(0), T, H,
        _ptr(q_norm_weight) if q_norm_weight is not None else None, float(eps), _ptr(kv), kv.stride(0),
        _ptr(positions), _ptr(slot_mapping), _ptr(cos_sin_cache), cos_sin_cache.shape[0], _ptr(kv_cache),
        kv_cache.numel() // 656, _stream(stream))


def dsv4_topk_select(scores: torch.Tensor, num_cand: torch.Tensor, top_k: int, topk_idx: torch.Tensor,
                     topk_lens: Optional[torch.Tensor] = None, stream=None) -> int:
    """scores float32 [T, width] (unit stride along a row); num_cand int32 [T];
    topk_idx int32 [T, top_k]; topk_lens int32 [T] or None."""
    _need(scores, torch.float32, "scores", 2)
    _need(num_cand, torch.int32, "num_cand", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    T, width = scores.shape
    return load_library().dsv4_topk_select(
        _ptr(scores) if width > 0 else None, max(scores.stride(0), width), width, _ptr(num_cand), T, int(top_k),
        _ptr(topk_idx), max(topk_idx.stride(0), topk_idx.shape[1]), _ptr(topk_lens) if topk_lens is not None else None,
        _stream(stream))


def dsv4_sparse_mla_decode_workspace_size(num_tokens: int, num_heads: int, topk_width: int, window: int) -> int:
    return int(load_library().dsv4_sparse_mla_decode_workspace_size(num_tokens, num_heads, topk_width, window))


def dsv4_sparse_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                           req_idx: Optional[torch.Tensor], topk_idx: torch.Tensor, topk_lens: Optional[torch.Tensor],
                           seq_lens: torch.Tensor, window: int, sink: Optional[torch.Tensor], softmax_scale: float,
                           out: torch.Tensor, lse: Optional[torch.Tensor], workspace: torch.Tensor,
                           stream=None) -> int:
    """q bf16 [T, H, 576] (heads contiguous); kv_cache uint8 [num_blocks, page, 656];
    block_table int32 [R, max_blocks]; req_idx int32 [T] or None; topk_idx int32 [T, K];
    topk_lens int32 [T] or None; seq_lens int32 [T]; sink float32 [H] or None;
    out bf16 [T, H, 512] contiguous; lse float32 [T, H] or None; workspace uint8 [>= workspace size]."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(req_idx, torch.int32, "req_idx", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(sink, torch.float32, "sink", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    _need(workspace, torch.uint8, "workspace", 1)
    if q.stride(1) != 576 or not kv_cache.is_contiguous() or not out.is_contiguous():
        raise ValueError("q heads must be contiguous rows of 576; kv_cache and out must be contiguous")
    if kv_cache.shape[2] != 656:
        raise ValueError("kv_cache entries must be 656 bytes")
    T, H, _ = q.shape
    K = topk_idx.shape[1]
    return load_library().dsv4_sparse_mla_decode(
        _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
        block_table.stride(0), block_table.shape[1], block_table.shape[0], _ptr(req_idx),
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(topk_lens), _ptr(seq_lens), T, H,
        int(window), _ptr(sink), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream))


def dsv4_sparse_mla_decode_trace(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                                 req_idx: Optional[torch.Tensor], topk_idx: torch.Tensor,
                                 topk_lens: Optional[torch.Tensor], seq_lens: torch.Tensor, window: int,
                                 sink: Optional[torch.Tensor], softmax_scale: float, out: torch.Tensor,
                                 lse: Optional[torch.Tensor], workspace: torch.Tensor, combined: torch.Tensor,
                                 combined_lens: torch.Tensor, stream=None) -> int:
    """dsv4_sparse_mla_decode that also records the combined list the decode kernel built:
    combined int32 [T, C] (C >= K + window) gets each token's positions [0, L), combined_lens
    int32 [T] gets L (see include/dsv4.h)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(req_idx, torch.int32, "req_idx", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(sink, torch.float32, "sink", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    _need(workspace, torch.uint8, "workspace", 1)
    _need(combined, torch.int32, "combined", 2)
    _need(combined_lens, torch.int32, "combined_lens", 1)
    if q.stride(1) != 576 or not kv_cache.is_contiguous() or not out.is_contiguous():
        raise ValueError("q heads must be contiguous rows of 576; kv_cache and out must be contiguous")
    if kv_cache.shape[2] != 656:
        raise ValueError("kv_cache entries must be 656 bytes")
    T, H, _ = q.shape
    K = topk_idx.shape[1]
    return load_library().dsv4_sparse_mla_decode_trace(
        _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
        block_table.stride(0), block_table.shape[1], block_table.shape[0], _ptr(req_idx),
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(topk_lens), _ptr(seq_lens), T, H,
        int(window), _ptr(sink), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _ptr(combined), max(combined.stride(0), combined.shape[1]), combined.shape[1], _ptr(combined_lens),
        _stream(stream))


def dsv4_sparse_mla_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                                   req_idx: Optional[torch.Tensor], topk_idx: torch.Tensor,
                                   topk_lens: Optional[torch.Tensor], seq_lens: torch.Tensor, window: int,
                                   sink: Optional[torch.Tensor], softmax_scale: float, out: torch.Tensor,
                                   lse: Optional[torch.Tensor], stream=None) -> int:
    """dsv4_sparse_mla_decode for callers that cannot allocate a workspace: the library's
    own 32 MiB static device array serves as scratch (see include/dsv4.h)."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(req_idx, torch.int32, "req_idx", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(sink, torch.float32, "sink", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    if q.stride(1) != 576 or not kv_cache.is_contiguous() or not out.is_contiguous():
        raise ValueError("q heads must be contiguous rows of 576; kv_cache and out must be contiguous")
    if kv_cache.shape[2] != 656:
        raise ValueError("kv_cache entries must be 656 bytes")
    T, H, _ = q.shape
    K = topk_idx.shape[1]
    return load_library().dsv4_sparse_mla_decode_noalloc(
        _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
        block_table.stride(0), block_table.shape[1], block_table.shape[0], _ptr(req_idx),
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(topk_lens), _ptr(seq_lens), T, H,
        int(window), _ptr(sink), float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream))


def dsv4_sparse_mla_decode_mtp_union_workspace_size(num_tokens: int, num_heads: int, topk_width: int,
                                                    window: int) -> int:
    return int(load_library().dsv4_sparse_mla_decode_mtp_union_workspace_size(num_tokens, num_heads, topk_width,
                                                                              window))


def dsv4_sparse_mla_decode_mtp_union(q: torch.Tensor, kv_cache: torch.Tensor, block_table: torch.Tensor,
                                     req_idx: torch.Tensor, topk_idx: torch.Tensor,
                                     topk_lens: Optional[torch.Tensor], seq_lens: torch.Tensor, window: int,
                                     sink: Optional[torch.Tensor], softmax_scale: float, out: torch.Tensor,
                                     lse: Optional[torch.Tensor], workspace: torch.Tensor, stream=None) -> int:
    """dsv4_sparse_mla_decode for batches of two-token requests (tokens 2r, 2r + 1 share
    req_idx[2r]) run over the union of each request's two key lists (see include/dsv4.h);
    workspace uint8 [>= dsv4_sparse_mla_decode_mtp_union_workspace_size(...)]."""
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(req_idx, torch.int32, "req_idx", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(topk_lens, torch.int32, "topk_lens", 1)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(sink, torch.float32, "sink", 1)
    _need(out, torch.bfloat16, "out", 3)
    _need(lse, torch.float32, "lse", 2)
    _need(workspace, torch.uint8, "workspace", 1)
    if q.stride(1) != 576 or not kv_cache.is_contiguous() or not out.is_contiguous():
        raise ValueError("q heads must be contiguous rows of 576; kv_cache and out must be contiguous")
    if kv_cache.shape[2] != 656:
        raise ValueError("kv_cache entries must be 656 bytes")
    T, H, _ = q.shape
    K = topk_idx.shape[1]
    return load_library().dsv4_sparse_mla_decode_mtp_union(
        _ptr(q), q.stride(0), _ptr(kv_cache), kv_cache.shape[0], kv_cache.shape[1], _ptr(block_table),
        block_table.stride(0), block_table.shape[1], block_table.shape[0], _ptr(req_idx),
        _ptr(topk_idx) if K > 0 else None, max(topk_idx.stride(0), K), K, _ptr(topk_lens), _ptr(seq_lens), T, H,
        int(window), _ptr(sink), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream))


def dsv4_get_device_status(stream=None) -> int:
    return int(load_library().dsv4_get_device_status(_stream(stream)))


# ----------------------------------------------------------------------------
# convenience: allocate outputs + workspace with torch, raise on error
# ----------------------------------------------------------------------------
def workspace_for(num_tokens: int, num_heads: int, topk_width: int, window: int, device=None) -> torch.Tensor:
    n = dsv4_sparse_mla_decode_workspace_size(num_tokens, num_heads, topk_width, window)
    if n == 0:
        raise Dsv4Error(DSV4_ERR_INVALID_ARG, "workspace size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def workspace_for_mtp_union(num_tokens: int, num_heads: int, topk_width: int, window: int, device=None) -> torch.Tensor:
    n = dsv4_sparse_mla_decode_mtp_union_workspace_size(num_tokens, num_heads, topk_width, window)
    if n == 0:
        raise Dsv4Error(DSV4_ERR_INVALID_ARG, "workspace size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def sparse_mla_decode(q, kv_cache, block_table, req_idx, topk_idx, topk_lens, seq_lens, window, sink,
                      softmax_scale, out=None, lse=None, workspace=None, stream=None):
    """Allocating wrapper of dsv4_sparse_mla_decode; returns (out, lse)."""
    T, H, _ = q.shape
    if out is None:
        out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(T, H, topk_idx.shape[1], window, q.device)
    check(dsv4_sparse_mla_decode(q, kv_cache, block_table, req_idx, topk_idx, topk_lens, seq_lens, window, sink,
                                 softmax_scale, out, lse, workspace, stream), "dsv4_sparse_mla_decode")
    return out, lse


def combine_topk_swa_indices(topk_idx, topk_lens, seq_lens, window, combined_width=None, stream=None):
    """Allocating wrapper of dsv4_combine_topk_swa_indices; returns (combined, combined_lens)."""
    T, K = topk_idx.shape
    if combined_width is None:
        combined_width = (K + window + 127) // 128 * 128
    combined = torch.empty((T, combined_width), dtype=torch.int32, device=seq_lens.device)
    lens = torch.empty((T,), dtype=torch.int32, device=seq_lens.device)
    check(dsv4_combine_topk_swa_indices(topk_idx, topk_lens, seq_lens, window, combined, lens, stream),
          "dsv4_combine_topk_swa_indices")
    return combined, lens
