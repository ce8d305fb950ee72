"""Thin Python binding of libsmla.so: argument marshalling only.

Every function forwards device pointers of torch tensors and the current CUDA
stream to the C entry point of the same name (include/smla.h) and raises
``SmlaError`` on a non-zero status.  All computation happens in the library's
CUDA kernels; there is no Python or CPU fallback."""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _lib

DEFAULT_SCALE = 1.0 / math.sqrt(512)
NOPE = 448
QK = 512
ROW_BYTES = 584


class SmlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib.load()
        super().__init__(f"{where}: {lib.smla_status_string(status).decode()} ({status})")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SmlaError(status, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def make_params(batch: int, num_heads: int, topk: int, num_rows: int, kv_row_stride: int,
                softmax_scale: float = DEFAULT_SCALE) -> _lib.SmlaParams:
    return _lib.SmlaParams(batch, num_heads, topk, 0, num_rows, kv_row_stride, softmax_scale)


def _params_from(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                 softmax_scale: float) -> _lib.SmlaParams:
    if q.dim() != 3 or q.shape[2] != QK or q.dtype != torch.bfloat16:
        raise ValueError("q must be bf16 [B, H, 512]")
    if kv_cache.dim() != 2 or kv_cache.dtype != torch.uint8 or kv_cache.stride(1) != 1:
        raise ValueError("kv_cache must be uint8 [num_rows, stride>=584] with unit column stride")
    if indices.dim() != 2 or indices.dtype != torch.int32 or indices.shape[0] != q.shape[0]:
        raise ValueError("indices must be int32 [B, topk]")
    for name, t in (("q", q), ("indices", indices)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.is_cuda and kv_cache.is_cuda and indices.is_cuda):
        raise ValueError("q, kv_cache and indices must be CUDA tensors")
    B, H, _ = q.shape
    return make_params(B, H, indices.shape[1], kv_cache.shape[0], kv_cache.stride(0),
                       softmax_scale)


def smla_default_num_splits(params: _lib.SmlaParams) -> int:
    lib = _lib.load()
    n = ctypes.c_int32(0)
    _check(lib.smla_default_num_splits(ctypes.byref(params), ctypes.byref(n)),
           "smla_default_num_splits")
    return n.value


def smla_decode_plan(params: _lib.SmlaParams, num_splits: int = 0) -> Tuple[int, bool]:
    """(resolved split count, True if sparse_mla_decode merges the splits on chip)."""
    lib = _lib.load()
    S, fused = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.smla_decode_plan(ctypes.byref(params), num_splits, ctypes.byref(S),
                                ctypes.byref(fused)), "smla_decode_plan")
    return S.value, bool(fused.value)


def smla_workspace_size(params: _lib.SmlaParams, num_splits: int = 0) -> int:
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _check(lib.smla_workspace_size(ctypes.byref(params), num_splits, ctypes.byref(n)),
           "smla_workspace_size")
    return n.value


def sparse_mla_decode(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                      softmax_scale: float = DEFAULT_SCALE, out: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                      workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None
                      ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Whole decode step.  Returns (out bf16 [B, H, 448], lse fp32 [B, H])."""
    p = _params_from(q, kv_cache, indices, softmax_scale)
    B, H = p.batch, p.num_heads
    if out is None:
        out = torch.empty((B, H, NOPE), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = smla_workspace_size(p, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    lib = _lib.load()
    st = lib.sparse_mla_decode(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(out), _ptr(lse),
                               ctypes.byref(p), num_splits, _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sparse_mla_decode")
    return out, lse


def sparse_mla_decode_split(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                            num_splits: int, softmax_scale: float = DEFAULT_SCALE,
                            o_part: Optional[torch.Tensor] = None,
                            lse_part: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None
                            ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split kernel alone.  Returns (o_part fp32 [B, H, S, 448], lse_part fp32 [B, H, S])."""
    p = _params_from(q, kv_cache, indices, softmax_scale)
    B, H, S = p.batch, p.num_heads, num_splits
    if o_part is None:
        o_part = torch.empty((B, H, S, NOPE), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    lib = _lib.load()
    st = lib.sparse_mla_decode_split(_ptr(q), _ptr(kv_cache), _ptr(indices), ctypes.byref(p), S,
                                     _ptr(o_part), _ptr(lse_part), _stream(stream))
    _check(st, "sparse_mla_decode_split")
    return o_part, lse_part


def sparse_mla_combine(o_part: torch.Tensor, lse_part: torch.Tensor,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None
                       ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Combine kernel alone.  Returns (out bf16 [B, H, 448], lse fp32 [B, H])."""
    if o_part.dim() != 4 or o_part.shape[3] != NOPE or o_part.dtype != torch.float32:
        raise ValueError("o_part must be fp32 [B, H, S, 448]")
    if lse_part.shape != o_part.shape[:3] or lse_part.dtype != torch.float32:
        raise ValueError("lse_part must be fp32 [B, H, S]")
    if not (o_part.is_contiguous() and lse_part.is_contiguous()):
        raise ValueError("partials must be contiguous")
    B, H, S, _ = o_part.shape
    if out is None:
        out = torch.empty((B, H, NOPE), dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=o_part.device)
    lib = _lib.load()
    st = lib.sparse_mla_combine(_ptr(o_part), _ptr(lse_part), B, H, S, _ptr(out), _ptr(lse),
                                _stream(stream))
    _check(st, "sparse_mla_combine")
    return out, lse


def sparse_mla_decode_noalloc(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                              softmax_scale: float = DEFAULT_SCALE,
                              out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                              stream: Optional[torch.cuda.Stream] = None
                              ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Whole decode step with the split partials in the library's built-in scratch
    (no workspace argument; the C function allocates nothing).  Pass `out` and `lse`
    to keep the call itself free of allocations."""
    p = _params_from(q, kv_cache, indices, softmax_scale)
    if out is None:
        out = torch.empty((p.batch, p.num_heads, NOPE), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_heads), dtype=torch.float32, device=q.device)
    st = _lib.load().sparse_mla_decode_noalloc(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(out),
                                               _ptr(lse), ctypes.byref(p), num_splits,
                                               _stream(stream))
    _check(st, "sparse_mla_decode_noalloc")
    return out, lse


def smla_paged_workspace_size(params: _lib.SmlaParams, num_splits: int = 0) -> int:
    lib = _lib.load()
    n = ctypes.c_size_t(0)
    _check(lib.smla_paged_workspace_size(ctypes.byref(params), num_splits, ctypes.byref(n)),
           "smla_paged_workspace_size")
    return n.value


def sparse_mla_decode_paged(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                            page_size: int, indices: torch.Tensor,
                            softmax_scale: float = DEFAULT_SCALE,
                            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                            num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None
                            ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Decode step over a paged cache: `indices` are logical positions in each query's
    sequence, `block_table` int32 [B, max_pages] maps its pages into `kv_pages`."""
    p = _params_from(q, kv_pages, indices, softmax_scale)
    if (block_table.dim() != 2 or block_table.dtype != torch.int32
            or block_table.shape[0] != p.batch or not block_table.is_contiguous()
            or not block_table.is_cuda):
        raise ValueError("block_table must be a contiguous CUDA int32 [B, max_pages] tensor")
    if out is None:
        out = torch.empty((p.batch, p.num_heads, NOPE), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_heads), dtype=torch.float32, device=q.device)
    need = smla_paged_workspace_size(p, num_splits)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = _lib.load().sparse_mla_decode_paged(
        _ptr(q), _ptr(kv_pages), _ptr(block_table), block_table.shape[1], page_size,
        _ptr(indices), _ptr(out), _ptr(lse), ctypes.byref(p), num_splits, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "sparse_mla_decode_paged")
    return out, lse


def sparse_mla_decode_simt(q: torch.Tensor, kv_cache: torch.Tensor, indices: torch.Tensor,
                           softmax_scale: float = DEFAULT_SCALE,
                           out: Optional[torch.Tensor] = None,
                           lse: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None
                           ) -> Tuple[torch.Tensor, torch.Tensor]:
    """The per-head fp32 SIMT form of the decode step (a reference point for the
    tensor-core path).  Returns (out bf16 [B, H, 448], lse fp32 [B, H])."""
    p = _params_from(q, kv_cache, indices, softmax_scale)
    if out is None:
        out = torch.empty((p.batch, p.num_heads, NOPE), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_heads), dtype=torch.float32, device=q.device)
    st = _lib.load().sparse_mla_decode_simt(_ptr(q), _ptr(kv_cache), _ptr(indices), _ptr(out),
                                            _ptr(lse), ctypes.byref(p), _stream(stream))
    _check(st, "sparse_mla_decode_simt")
    return out, lse


def smla_device_status(clear: bool = False) -> int:
    """Device status word (0, SMLA_ERR_TIMEOUT or SMLA_ERR_INDEX_RANGE); synchronises."""
    lib = _lib.load()
    v = ctypes.c_int32(0)
    _check(lib.smla_device_status(ctypes.byref(v), 1 if clear else 0), "smla_device_status")
    return v.value


def smla_status_string(status: int) -> str:
    return _lib.load().smla_status_string(status).decode()
