"""lightning_indexer_top_gb300 -- lightning-indexer sparse attention on GB300.

A thin ctypes binding over ``liblidx.so`` (C ABI in ``include/lidx.h``).  The
functions here only marshal torch tensors into pointers, sizes and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no CPU fallback: if the library is missing or fails to load, every
call raises.

Build with ``lightning_indexer_top_gb300.build()`` (nvcc, sm_103a).
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

from ._build import LIB as _LIB_PATH
from ._build import build  # noqa: F401

__all__ = [
    "Batch", "LidxError", "build", "load", "idx_hadamard", "idx_score", "idx_block_pool", "idx_block_pool_update",
    "idx_quantize_rows", "idx_score_q8", "inline_scales",
    "idx_topk", "sparse_attn_decode", "sparse_attn_prefill", "idx_workspace_size",
    "idx_device_status", "topk_capacity", "sparse_attn_decode_noalloc", "idx_score_topk", "idx_block_score_topk", "sparse_decode_step", "sparse_decode_step_fused",
]

IDX_OK, IDX_ERR_INVALID_ARG, IDX_ERR_UNSUPPORTED, IDX_ERR_CUDA, IDX_ERR_TIMEOUT, IDX_ERR_DEVICE_BOUNDS, IDX_ERR_INEXACT = range(7)
IDX_F32, IDX_F16, IDX_BF16 = 0, 1, 2
IDX_POS_CLEAN = 2**31 - 1   # stale_pos value: no edit
IDX_OP_SCORE, IDX_OP_TOPK, IDX_OP_ATTN_DECODE, IDX_OP_ATTN_PREFILL, IDX_OP_SCORE_TOPK, IDX_OP_DECODE_STEP = 0, 1, 2, 3, 4, 5

_DTYPES = {torch.float32: IDX_F32, torch.float16: IDX_F16, torch.bfloat16: IDX_BF16}


class LidxError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"lidx status {status}: {msg}")
        self.status = status


class _Batch(ctypes.Structure):
    _fields_ = [
        ("n_seq", ctypes.c_int32),
        ("n_q_per_seq", ctypes.c_int32),
        ("n_kv", ctypes.c_void_p),
        ("kv_start", ctypes.c_void_p),
        ("kv_seq_stride", ctypes.c_int64),
        ("q_pos", ctypes.c_void_p),
        ("max_n_kv", ctypes.c_int32),
        ("page_table", ctypes.c_void_p),
        ("page_table_stride", ctypes.c_int64),
        ("page_size", ctypes.c_int32),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load liblidx.so (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run lightning_indexer_top_gb300.build() first")
    lib = ctypes.CDLL(path)
    P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sigs = {
        "idx_hadamard": [P, P, I32, I64, I32, I64, P],
        "idx_score": [P, I32, P, I32, I32, P, I32, I64, I64, _Batch, I32, P, I64, P, SZ, P],
        "idx_block_pool": [P, I32, I64, I64, _Batch, I32, I32, P, I64, P],
        "idx_block_pool_update": [P, I32, I64, I64, _Batch, P, P, I32, I32, P, I64, P],
        "idx_quantize_rows": [P, I32, I64, I32, I64, P, I64, P, P],
        "idx_score_q8": [P, I32, P, I32, I32, P, I64, P, I64, _Batch, I32, P, I64, P, SZ, P],
        "idx_topk": [P, I64, _Batch, I32, I32, P, I64, P, P, SZ, P],
        "idx_score_topk": [P, I32, P, I32, I32, P, I32, I64, I64, _Batch, I32, P, I64, P, I64, P, P, SZ, P],
        "idx_block_score_topk": [P, I32, P, I32, I32, P, I32, I64, I64, _Batch, P, P, I32, P, I64, I32, P, I64, P,
                                 I64, P, P],
        "sparse_attn_decode": [P, I32, I32, I32, I32, I32, P, P, I64, I64, I64, _Batch, P, I64, P, F,
                               P, I32, P, SZ, P],
        "sparse_attn_prefill": [P, I32, I32, I32, I32, I32, P, P, I64, I64, I64, _Batch, P, I64, P, F,
                                P, I32, P, SZ, P],
        "sparse_attn_decode_noalloc": [P, I32, I32, I32, I32, I32, P, I64, I64, _Batch, P, I64, P, F, P, I32, P],
        "sparse_decode_step": [P, I32, P, I32, I32, P, I32, I64, I64, _Batch, I32, P, I64, P, I64, P,
                               P, I32, I32, I32, I32, I32, P, P, I64, I64, I64, F, P, I32, P, SZ, P],
        "idx_workspace_size": [I32, I64, I32, I32, I32, I32],
        "sparse_decode_step_fused": [I64, I32, I32, I32, I64],
        "idx_last_error": [],
        "idx_device_status": [I32],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.idx_workspace_size.restype = ctypes.c_size_t
    lib.idx_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != IDX_OK:
        raise LidxError(status, load().idx_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("lidx operates on CUDA tensors only")


@dataclass
class Batch:
    """Batch geometry (see idx_batch in include/lidx.h).

    n_kv:      int32 CUDA tensor [B], cached tokens per sequence.
    n_q_per_seq: query rows per sequence (decode: 1).
    max_n_kv:  host bound on every n_kv[b].
    kv_start:  optional int32 CUDA tensor [B]: cache row of position 0.
    kv_seq_stride: rows between sequences when kv_start is None.
    q_pos:     optional int32 CUDA tensor [B*T]: causal position per query row.
    page_table: optional int32 CUDA tensor [B, pages]: physical page of each logical page
               (position j of sequence b is cache row page_table[b, j // page_size] * page_size
               + j % page_size); kv_start / kv_seq_stride are then unused.
    """

    n_kv: torch.Tensor
    n_q_per_seq: int
    max_n_kv: int
    kv_start: Optional[torch.Tensor] = None
    kv_seq_stride: int = 0
    q_pos: Optional[torch.Tensor] = None
    page_table: Optional[torch.Tensor] = None
    page_size: int = 0

    @property
    def n_seq(self) -> int:
        return int(self.n_kv.numel())

    @property
    def n_rows(self) -> int:
        return self.n_seq * self.n_q_per_seq

    def c(self) -> _Batch:
        for t in (self.n_kv, self.kv_start, self.q_pos, self.page_table):
            if t is not None and (t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous()):
                raise ValueError("batch arrays must be contiguous int32 CUDA tensors")
        pt_stride = self.page_table.shape[-1] if self.page_table is not None else 0
        return _Batch(self.n_seq, self.n_q_per_seq, _ptr(self.n_kv), _ptr(self.kv_start),
                      self.kv_seq_stride, _ptr(self.q_pos), self.max_n_kv, _ptr(self.page_table), pt_stride,
                      self.page_size if self.page_table is not None else 0)


IDX_DEFAULT_TOP_K = 2048   # top_k = -1: the model's configured indexer top_k


def topk_capacity(top_k: int, block_size: int = 0) -> int:
    """Row capacity idx_topk writes: top_k, or floor(top_k/C)*C + C - 1 in block mode (-1: the default)."""
    if top_k == -1:
        top_k = IDX_DEFAULT_TOP_K
    if block_size > 1:
        return (top_k // block_size) * block_size + block_size - 1
    return top_k


def idx_hadamard(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Rotate the rows (last dim) of x by the orthonormal Hadamard matrix into `out`
    (in place when out is None or is x)."""
    out = x if out is None else out
    _need_cuda(x, out)
    if not x.is_contiguous() or not out.is_contiguous() or out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("x and out must be contiguous tensors of the same shape and dtype")
    d = x.shape[-1]
    rows = x.numel() // d
    _check(load().idx_hadamard(_ptr(x), _ptr(out), _dtype(x), rows, d, d, _stream(x.device)))
    return out


def idx_workspace_size(op: int, n_rows: int, max_n_kv: int, top_k: int, n_q_heads: int = 0, dv: int = 0) -> int:
    return int(load().idx_workspace_size(op, n_rows, max_n_kv, top_k, n_q_heads, dv))


def idx_score(q: torch.Tensor, w: torch.Tensor, k: torch.Tensor, batch: Batch, *, block_size: int = 0,
              scores: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Indexer scores [B*T, keys] f32.  q [B*T, H, d]; w [B*T, H] f32; k [rows, d] (key cache
    or pooled keys when block_size > 1)."""
    _need_cuda(q, w, k, scores, workspace)
    rows, H, d = q.shape
    assert rows == batch.n_rows and w.shape == (rows, H) and w.dtype == torch.float32
    assert q.is_contiguous() and w.is_contiguous() and k.stride(-1) == 1
    keys = batch.max_n_kv // block_size if block_size > 1 else batch.max_n_kv
    if scores is None:
        scores = torch.empty(rows, max(keys, 1), device=q.device, dtype=torch.float32)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().idx_score(_ptr(q), _dtype(q), _ptr(w), H, d, _ptr(k), _dtype(k), k.stride(0),
                            k.shape[0], batch.c(), block_size, _ptr(scores), scores.stride(0),
                            _ptr(workspace), ws_bytes, _stream(q.device)))
    return scores


def idx_block_pool(k_raw: torch.Tensor, batch: Batch, block_size: int, *, pool_seq_stride: Optional[int] = None,
                   pooled: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Mean-pooled complete blocks, f32 [B, pool_seq_stride, d]."""
    _need_cuda(k_raw, pooled)
    d = k_raw.shape[-1]
    if pool_seq_stride is None:
        pool_seq_stride = max(batch.max_n_kv // block_size, 1)
    if pooled is None:
        pooled = torch.zeros(batch.n_seq, pool_seq_stride, d, device=k_raw.device, dtype=torch.float32)
    _check(load().idx_block_pool(_ptr(k_raw), _dtype(k_raw), k_raw.stride(0), k_raw.shape[0], batch.c(),
                                 block_size, d, _ptr(pooled), pool_seq_stride, _stream(k_raw.device)))
    return pooled


def idx_quantize_rows(x: torch.Tensor, *, q8: Optional[torch.Tensor] = None,
                      scale: Optional[torch.Tensor] = None, inline_scale: bool = False):
    """Per-row int8 codes and f32 scales of key rows [n, d]: x ~= scale[:, None] * q8.

    inline_scale: each row's scale is stored in bytes d .. d+3 of its code row (rows of
    ceil((d + 4) / 16) * 16 bytes); returns (rows [n, that width] int8, None)."""
    _need_cuda(x, q8, scale)
    n, d = x.shape[0], x.shape[-1]
    if inline_scale:
        if q8 is None:
            q8 = torch.empty(n, (d + 4 + 15) // 16 * 16, device=x.device, dtype=torch.int8)
        _check(load().idx_quantize_rows(_ptr(x), _dtype(x), n, d, x.stride(0), _ptr(q8), q8.stride(0), None,
                                        _stream(x.device)))
        return q8, None
    if q8 is None:
        q8 = torch.empty(n, (d + 15) // 16 * 16, device=x.device, dtype=torch.int8)[:, :d]
    if scale is None:
        scale = torch.empty(n, device=x.device, dtype=torch.float32)
    _check(load().idx_quantize_rows(_ptr(x), _dtype(x), n, d, x.stride(0), _ptr(q8), q8.stride(0), _ptr(scale),
                                    _stream(x.device)))
    return q8, scale


def inline_scales(rows: torch.Tensor, d: int) -> torch.Tensor:
    """The f32 scales stored inline (bytes d .. d+3) in int8 code rows written with inline_scale."""
    return rows[:, d:d + 4].contiguous().view(torch.float32).view(-1)


def idx_score_q8(q: torch.Tensor, w: torch.Tensor, k8: torch.Tensor, k_scale: Optional[torch.Tensor],
                 batch: Batch, *, scores: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Indexer scores over an int8 key cache with per-row scales (f32 [rows, keys]);
    k_scale None: the scales are inline in the rows (idx_quantize_rows(..., inline_scale=True))."""
    _need_cuda(q, w, k8, k_scale, scores)
    H, d = q.shape[-2], q.shape[-1]
    rows = batch.n_rows
    if scores is None:
        scores = torch.empty(rows, max(batch.max_n_kv, 1), device=q.device, dtype=torch.float32)
    _check(load().idx_score_q8(_ptr(q), _dtype(q), _ptr(w), H, d, _ptr(k8), k8.stride(0), _ptr(k_scale),
                               k8.shape[0], batch.c(), 0, _ptr(scores), scores.stride(0), None, 0,
                               _stream(q.device)))
    return scores


def idx_block_pool_update(k_raw: torch.Tensor, batch: Batch, block_size: int, pooled: torch.Tensor, *,
                          n_pooled: Optional[torch.Tensor] = None, stale_pos: Optional[torch.Tensor] = None,
                          pool_seq_stride: Optional[int] = None) -> torch.Tensor:
    """(Re)pool only the blocks from min(n_pooled[b], stale_pos[b] // C) on, in place in ``pooled``.

    n_pooled / stale_pos: device int32 [n_seq] or None (0 / no edit); IDX_POS_CLEAN marks no edit.
    """
    _need_cuda(k_raw, pooled, n_pooled, stale_pos)
    d = k_raw.shape[-1]
    if pool_seq_stride is None:
        pool_seq_stride = pooled.shape[1] if pooled.dim() == 3 else max(batch.max_n_kv // block_size, 1)
    for t in (n_pooled, stale_pos):
        if t is not None and (t.dtype != torch.int32 or t.numel() < batch.n_seq or not t.is_contiguous()):
            raise ValueError("n_pooled / stale_pos must be contiguous int32 with one entry per sequence")
    _check(load().idx_block_pool_update(_ptr(k_raw), _dtype(k_raw), k_raw.stride(0), k_raw.shape[0], batch.c(),
                                        _ptr(n_pooled), _ptr(stale_pos), block_size, d, _ptr(pooled),
                                        pool_seq_stride, _stream(k_raw.device)))
    return pooled


def idx_topk(scores: torch.Tensor, batch: Batch, top_k: int, *, block_size: int = 0,
             idx: Optional[torch.Tensor] = None, n_sel: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None):
    """Selected positions (ascending, -1 padded) and their count per row."""
    _need_cuda(scores, idx, n_sel, workspace)
    rows = batch.n_rows
    cap = topk_capacity(top_k, block_size)
    if idx is None:
        idx = torch.empty(rows, cap, device=scores.device, dtype=torch.int32)
    if n_sel is None:
        n_sel = torch.empty(rows, device=scores.device, dtype=torch.int32)
    if workspace is None and block_size <= 1:
        need = idx_workspace_size(IDX_OP_TOPK, rows, batch.max_n_kv, top_k)
        if need:
            workspace = torch.empty(need, device=scores.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().idx_topk(_ptr(scores), scores.stride(0), batch.c(), top_k, block_size, _ptr(idx),
                           idx.stride(0), _ptr(n_sel), _ptr(workspace), ws_bytes, _stream(scores.device)))
    return idx, n_sel


def _attn(fn_name, q, k, v, batch, idx, n_sel, scale, out, out_dtype, workspace, n_kv_heads, dv):
    _need_cuda(q, k, v, idx, n_sel, out, workspace)
    rows, Hq, dk = q.shape
    assert rows == batch.n_rows and q.is_contiguous()
    if v is None:
        hkv, dv = 1, (dv if dv is not None else 512)
        kv_row_stride = k.stride(0)
        v_row_stride = 0
    else:
        hkv = n_kv_heads if n_kv_heads is not None else k.shape[1]
        dv = v.shape[-1]
        kv_row_stride = k.stride(0)
        v_row_stride = v.stride(0)
    if out is None:
        out = torch.empty(rows, Hq, dv, device=q.device, dtype=out_dtype)
    if workspace is None:
        op = IDX_OP_ATTN_PREFILL if fn_name == "sparse_attn_prefill" else IDX_OP_ATTN_DECODE
        need = idx_workspace_size(op, rows, batch.max_n_kv, idx.stride(0), Hq, dv)
        if need:
            workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = getattr(load(), fn_name)
    _check(fn(_ptr(q), _dtype(q), Hq, hkv, dk, dv, _ptr(k), _ptr(v), kv_row_stride, v_row_stride,
              k.shape[0], batch.c(), _ptr(idx), idx.stride(0), _ptr(n_sel), float(scale), _ptr(out),
              _dtype(out), _ptr(workspace), ws_bytes, _stream(q.device)))
    return out


def sparse_attn_decode(q, k, v, batch, idx, n_sel, scale, *, out=None, out_dtype=torch.float32,
                       workspace=None, n_kv_heads=None, dv=None):
    """Attention over the selected keys.  q [B*T, Hq, dk]; k [rows, Hkv, dk] (or the MLA latent
    [rows, 576] with v=None and dv=512); v [rows, Hkv, dv] or None."""
    return _attn("sparse_attn_decode", q, k, v, batch, idx, n_sel, scale, out, out_dtype, workspace,
                 n_kv_heads, dv)


def sparse_attn_prefill(q, k, v, batch, idx, n_sel, scale, *, out=None, out_dtype=torch.float32,
                        workspace=None, n_kv_heads=None, dv=None):
    """Same function as sparse_attn_decode, tuned for many query rows."""
    return _attn("sparse_attn_prefill", q, k, v, batch, idx, n_sel, scale, out, out_dtype, workspace,
                 n_kv_heads, dv)


def idx_block_score_topk(q: torch.Tensor, w: torch.Tensor, k_raw: torch.Tensor, batch: Batch, block_size: int,
                         pooled: torch.Tensor, top_k: int, *, n_pooled: Optional[torch.Tensor] = None,
                         stale_pos: Optional[torch.Tensor] = None, pool_seq_stride: Optional[int] = None,
                         scores: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                         n_sel: Optional[torch.Tensor] = None):
    """The indexer of a block-pooled decode step in one call: (scores, idx, n_sel) exactly as
    idx_block_pool_update + idx_score over ``pooled`` + idx_topk in block mode give them; ``pooled``
    is updated in place."""
    _need_cuda(q, w, k_raw, pooled, n_pooled, stale_pos, scores, idx, n_sel)
    rows, H, d = q.shape
    assert rows == batch.n_rows and w.shape == (rows, H) and w.dtype == torch.float32
    assert q.is_contiguous() and w.is_contiguous() and k_raw.stride(-1) == 1
    assert pooled.dtype == torch.float32 and pooled.is_contiguous()
    if pool_seq_stride is None:
        pool_seq_stride = pooled.shape[1] if pooled.dim() == 3 else max(batch.max_n_kv // block_size, 1)
    for t in (n_pooled, stale_pos):
        if t is not None and (t.dtype != torch.int32 or t.numel() < batch.n_seq or not t.is_contiguous()):
            raise ValueError("n_pooled / stale_pos must be contiguous int32 with one entry per sequence")
    kk = 2048 if top_k == -1 else top_k
    if scores is None:
        scores = torch.empty(rows, max(batch.max_n_kv // block_size, 1), device=q.device, dtype=torch.float32)
    if idx is None:
        idx = torch.empty(rows, topk_capacity(kk, block_size), device=q.device, dtype=torch.int32)
    if n_sel is None:
        n_sel = torch.empty(rows, device=q.device, dtype=torch.int32)
    _check(load().idx_block_score_topk(_ptr(q), _dtype(q), _ptr(w), H, d, _ptr(k_raw), _dtype(k_raw), k_raw.stride(0),
                                       k_raw.shape[0], batch.c(), _ptr(n_pooled), _ptr(stale_pos), block_size,
                                       _ptr(pooled), pool_seq_stride, top_k, _ptr(scores), scores.stride(0), _ptr(idx),
                                       idx.stride(0), _ptr(n_sel), _stream(q.device)))
    return scores, idx, n_sel


def idx_score_topk(q: torch.Tensor, w: torch.Tensor, k: torch.Tensor, batch: Batch, top_k: int, *,
                   scores: Optional[torch.Tensor] = None, idx: Optional[torch.Tensor] = None,
                   n_sel: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """The fused indexer + selection (token keys): (scores, idx, n_sel) exactly as idx_score followed
    by idx_topk would give them."""
    _need_cuda(q, w, k, scores, idx, n_sel, workspace)
    rows, H, d = q.shape
    assert rows == batch.n_rows and w.shape == (rows, H) and w.dtype == torch.float32
    assert q.is_contiguous() and w.is_contiguous() and k.stride(-1) == 1
    kk = 2048 if top_k == -1 else top_k
    if scores is None:
        scores = torch.empty(rows, max(batch.max_n_kv, 1), device=q.device, dtype=torch.float32)
    if idx is None:
        idx = torch.empty(rows, kk, device=q.device, dtype=torch.int32)
    if n_sel is None:
        n_sel = torch.empty(rows, device=q.device, dtype=torch.int32)
    if workspace is None:
        need = idx_workspace_size(IDX_OP_SCORE_TOPK, rows, batch.max_n_kv, top_k)
        if need:
            workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().idx_score_topk(_ptr(q), _dtype(q), _ptr(w), H, d, _ptr(k), _dtype(k), k.stride(0), k.shape[0],
                                 batch.c(), top_k, _ptr(scores), scores.stride(0), _ptr(idx), idx.stride(0),
                                 _ptr(n_sel), _ptr(workspace), ws_bytes, _stream(q.device)))
    return scores, idx, n_sel


def sparse_decode_step(q: torch.Tensor, w: torch.Tensor, k: torch.Tensor, batch: Batch, top_k: int,
                       q_attn: torch.Tensor, k_attn: torch.Tensor, v_attn: Optional[torch.Tensor], scale: float, *,
                       dv: Optional[int] = None, scores: Optional[torch.Tensor] = None,
                       idx: Optional[torch.Tensor] = None, n_sel: Optional[torch.Tensor] = None,
                       out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                       workspace: Optional[torch.Tensor] = None):
    """One decode step: idx_score_topk then sparse_attn_decode (one launch for few short rows).
    Returns (scores, idx, n_sel, out)."""
    _need_cuda(q, w, k, q_attn, k_attn, v_attn, scores, idx, n_sel, out, workspace)
    rows, H, d = q.shape
    assert rows == batch.n_rows and w.shape == (rows, H) and w.dtype == torch.float32
    assert q.is_contiguous() and w.is_contiguous() and k.stride(-1) == 1 and q_attn.is_contiguous()
    _, Hq, dk = q_attn.shape
    if v_attn is None:
        hkv, dv = 1, (dv if dv is not None else 512)
        v_row_stride = 0
    else:
        hkv, dv = k_attn.shape[1], v_attn.shape[-1]
        v_row_stride = v_attn.stride(0)
    kk = 2048 if top_k == -1 else top_k
    if scores is None:
        scores = torch.empty(rows, max(batch.max_n_kv, 1), device=q.device, dtype=torch.float32)
    if idx is None:
        idx = torch.empty(rows, kk, device=q.device, dtype=torch.int32)
    if n_sel is None:
        n_sel = torch.empty(rows, device=q.device, dtype=torch.int32)
    if out is None:
        out = torch.empty(rows, Hq, dv, device=q.device, dtype=out_dtype)
    if workspace is None:
        need = idx_workspace_size(IDX_OP_DECODE_STEP, rows, batch.max_n_kv, top_k, Hq, dv)
        if need:
            workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sparse_decode_step(_ptr(q), _dtype(q), _ptr(w), H, d, _ptr(k), _dtype(k), k.stride(0), k.shape[0],
                                     batch.c(), top_k, _ptr(scores), scores.stride(0), _ptr(idx), idx.stride(0),
                                     _ptr(n_sel), _ptr(q_attn), _dtype(q_attn), Hq, hkv, dk, dv, _ptr(k_attn),
                                     _ptr(v_attn), k_attn.stride(0), v_row_stride, k_attn.shape[0], float(scale),
                                     _ptr(out), _dtype(out), _ptr(workspace), ws_bytes, _stream(q.device)))
    return scores, idx, n_sel, out


def sparse_decode_step_fused(n_rows: int, n_q_per_seq: int, max_n_kv: int, top_k: int, idx_row_stride: int) -> bool:
    """Whether sparse_decode_step runs as one launch for these sizes on the current device."""
    return bool(load().sparse_decode_step_fused(n_rows, n_q_per_seq, max_n_kv, top_k, idx_row_stride))


def sparse_attn_decode_noalloc(q, latent, batch, idx, n_sel, scale, *, out=None, out_dtype=torch.bfloat16):
    """The 128-head MLA decode attention without a workspace, for callers that cannot
    allocate device memory: its key-split scratch is a static array inside the library
    (see include/lidx.h).  Calls that overlap on the GPU must be serialised."""
    _need_cuda(q, latent, idx, n_sel, out)
    rows, Hq, dk = q.shape
    assert rows == batch.n_rows and q.is_contiguous()
    if out is None:
        out = torch.empty(rows, Hq, 512, device=q.device, dtype=out_dtype)
    _check(load().sparse_attn_decode_noalloc(_ptr(q), _dtype(q), Hq, 1, dk, 512, _ptr(latent), latent.stride(0),
                                             latent.shape[0], batch.c(), _ptr(idx), idx.stride(0), _ptr(n_sel),
                                             float(scale), _ptr(out), _dtype(out), _stream(q.device)))
    return out


def idx_device_status(reset: bool = True) -> int:
    """Synchronise and return the device fault word (0 = none)."""
    return int(load().idx_device_status(1 if reset else 0))
