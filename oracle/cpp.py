"""The C++ oracle (lidx_oracle.cpp) behind the numpy oracle's function names.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This module only
marshals arrays into the C functions through ctypes: every step of the
arithmetic runs in lidx_oracle.cpp.  The single-row functions take the same
arguments and return the same types as their namesakes in lidx_oracle.py, so
that the pins in tests/test_oracle_pins.py run against both implementations;
the ``*_batch`` functions spread many query rows over the host cores (OpenMP)
and read large caches in their storage type (f16 / bf16 / int8), without
widening them in Python first.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np

from . import build_cpp

F64, F32, F16, BF16, I8 = 0, 1, 2, 3, 4
_FMT_NAMES = {"f64": F64, "f32": F32, "f16": F16, "bf16": BF16}

_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def lib():
    """Build (if stale) and load liblidx_oracle.so."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build_cpp.build())
        sig = {
            "oracle_threads": ([], ctypes.c_int),
            "oracle_round_storage": ([_P, _I64, _I32, _P], None),
            "oracle_widen": ([_P, _I32, _I64, _P], None),
            "oracle_hadamard_matrix": ([_I32, _P], None),
            "oracle_hadamard": ([_P, _I64, _I32, _I32, _P], None),
            "oracle_visible_count": ([_I64, _I32, _I64], _I64),
            "oracle_scores": ([_I64, _I32, _I32, _P, _I32, _P, _P, _I32, _I64, _P, _P, _P, _P, _I64], None),
            "oracle_topk": ([_I64, _P, _I64, _P, _I32, _P, _I64, _P], ctypes.c_int),
            "oracle_block_pool": ([_P, _I32, _I64, _I64, _I32, _I32, _P], None),
            "oracle_block_pool_update": ([_P, _I64, _P, _I32, _I64, _I64, _I32, _I32, _I64, _I32, _I64, _P], None),
            "oracle_block_select": ([_I64, _P, _I64, _P, _I32, _I32, _P, _I64, _P], ctypes.c_int),
            "oracle_block_select_expanded": ([_I64, _P, _I64, _P, _I32, _I32, _P, _I64, _P], ctypes.c_int),
            "oracle_attention": ([_I64, _I32, _I32, _I32, _I32, _P, _I32, _P, _I32, _I64, _P, _I32, _I64, _P, _P,
                                  _I64, _P, ctypes.c_double, _P], ctypes.c_int),
            "oracle_quantize_rows": ([_P, _I32, _I64, _I32, _I64, _P, _P], None),
            "oracle_dequantize_rows": ([_P, _P, _I64, _I32, _P], None),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def threads() -> int:
    """OpenMP threads the oracle uses (all host cores unless OMP_NUM_THREADS says otherwise)."""
    return int(lib().oracle_threads())


# ---------------------------------------------------------------- marshalling

def stored(x):
    """(contiguous numpy buffer, format code) of an array in its storage type.

    numpy float64 / float32 / float16 / int8 arrays keep their type; a torch
    tensor (any device) is copied to the host as it is stored, bfloat16 as its
    raw 16-bit patterns; anything else is taken as float64."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach().to("cpu").contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16), BF16
        if t.dtype == torch.float16:
            return t.numpy(), F16
        if t.dtype == torch.float32:
            return t.numpy(), F32
        if t.dtype == torch.int8:
            return t.numpy(), I8
        return t.to(torch.float64).numpy(), F64
    a = np.ascontiguousarray(x)
    fmt = {np.dtype(np.float64): F64, np.dtype(np.float32): F32, np.dtype(np.float16): F16,
           np.dtype(np.int8): I8}.get(a.dtype)
    if fmt is None:
        a, fmt = np.ascontiguousarray(a, dtype=np.float64), F64
    return a, fmt


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_P)


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float64)


# ---------------------------------------------------------------- storage rounding, Hadamard

def round_to_storage(x, fmt: str) -> np.ndarray:
    a = _f64(x)
    y = np.empty_like(a)
    lib().oracle_round_storage(_ptr(a), a.size, _FMT_NAMES[fmt], _ptr(y))
    return y


def hadamard_matrix(d: int) -> np.ndarray:
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.empty((d, d))
    lib().oracle_hadamard_matrix(d, _ptr(h))
    return h


def hadamard_rotate(x, store: str | None = None) -> np.ndarray:
    a = _f64(x)
    d = a.shape[-1]
    if d < 1 or d & (d - 1):
        raise ValueError("Hadamard order must be a power of two")
    y = np.empty_like(a)
    lib().oracle_hadamard(_ptr(a), a.size // d, d, _FMT_NAMES[store] if store else F64, _ptr(y))
    return y


def visible_count(n_kv: int, q_pos: int | None) -> int:
    return int(lib().oracle_visible_count(int(n_kv), 0 if q_pos is None else 1, 0 if q_pos is None else int(q_pos)))


# ---------------------------------------------------------------- scores

def scores_batch(q, w, k, key_off, n_vis, k_scale=None, out_cols=None) -> np.ndarray:
    """Scores of R query rows: row r scores keys key_off[r] .. key_off[r] + n_vis[r] - 1.

    q [R, H, d] and k [rows, d] in their storage types (k int8 with k_scale f32
    [rows] for a quantized cache), w [R, H].  Returns float32 [R, out_cols];
    entries past n_vis[r] are 0."""
    qa, qf = stored(q)
    ka, kf = stored(k)
    R, H, d = qa.shape
    wa = _f64(w).reshape(R, H)
    ko = np.ascontiguousarray(key_off, dtype=np.int64)
    nv = np.ascontiguousarray(n_vis, dtype=np.int32)
    cols = int(out_cols if out_cols is not None else (nv.max() if R else 0))
    out = np.zeros((R, max(cols, 1)), np.float32)
    sc = None
    if kf == I8:
        sc = np.ascontiguousarray(k_scale, dtype=np.float32)
    ka2 = ka.reshape(ka.shape[0], -1) if ka.ndim > 1 else ka.reshape(-1, d)
    lib().oracle_scores(R, H, d, _ptr(qa), qf, _ptr(wa), _ptr(ka2), kf, ka2.shape[1],
                        _ptr(sc) if sc is not None else None, _ptr(ko), _ptr(nv), _ptr(out), out.shape[1])
    return out[:, :cols]


def indexer_scores(q, w, k) -> np.ndarray:
    q = _f64(q)
    k = _f64(k)
    n = k.shape[0]
    if n == 0:
        return np.zeros(0, dtype=np.float32)
    return scores_batch(q[None], _f64(w)[None], k, [0], [n], out_cols=n)[0]


# ---------------------------------------------------------------- top-k

def topk_batch(scores, n_vis, top_k: int):
    """(idx int32 [R, top_k] ascending and -1 padded, n_sel int32 [R])."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    if s.ndim == 1:
        s = s[None]
    R = s.shape[0]
    nv = np.ascontiguousarray(n_vis, dtype=np.int32)
    cap = max(int(top_k), 1)
    idx = np.empty((R, cap), np.int32)
    ns = np.empty(R, np.int32)
    if lib().oracle_topk(R, _ptr(s), s.shape[1], _ptr(nv), int(top_k), _ptr(idx), cap, _ptr(ns)):
        raise ValueError("scores must be finite")
    return idx, ns


def topk_select(scores, n_vis: int, top_k: int) -> np.ndarray:
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float32)[:n_vis])
    kk = min(int(top_k), int(n_vis))
    if kk <= 0:
        if not np.all(np.isfinite(s)):
            raise ValueError("scores must be finite")
        return np.zeros(0, dtype=np.int64)
    idx, ns = topk_batch(s.reshape(1, -1) if s.size else np.zeros((1, 1), np.float32), [int(n_vis)], kk)
    return idx[0, :ns[0]].astype(np.int64)


# ---------------------------------------------------------------- blocks

def block_pool(k_raw, C: int, n_kv: int) -> np.ndarray:
    ka, kf = stored(k_raw)
    d = ka.shape[-1]
    ka = ka.reshape(-1, d)
    n_cb = int(n_kv) // int(C)
    out = np.zeros((n_cb, d), np.float32)
    if n_cb:
        lib().oracle_block_pool(_ptr(ka), kf, d, int(n_kv), int(C), d, _ptr(out))
    return out


def block_pool_update(pooled_prev, k_raw, C: int, n_kv: int, n_pooled: int, stale_pos=None) -> np.ndarray:
    prev = np.ascontiguousarray(pooled_prev, dtype=np.float32)
    ka, kf = stored(k_raw)
    d = prev.shape[-1]
    ka = ka.reshape(-1, d)
    out = np.empty_like(prev)
    lib().oracle_block_pool_update(_ptr(prev), prev.shape[0], _ptr(ka), kf, d, int(n_kv), int(C), d,
                                   int(n_pooled), 0 if stale_pos is None else 1,
                                   0 if stale_pos is None else int(stale_pos), _ptr(out))
    return out


def _block_select(fn, block_scores, n_vis, top_k, C):
    n_cb = int(n_vis) // int(C)
    bs = np.ascontiguousarray(np.asarray(block_scores, dtype=np.float32)[:n_cb])
    if bs.size == 0:
        bs = np.zeros(1, np.float32)
    cap = (int(top_k) // int(C)) * int(C) + int(C) - 1
    idx = np.empty(max(cap, 1), np.int32)
    ns = np.empty(1, np.int32)
    nv = np.array([int(n_vis)], np.int32)
    if fn(1, _ptr(bs), bs.size, _ptr(nv), int(top_k), int(C), _ptr(idx), idx.size, _ptr(ns)):
        raise ValueError("block scores must be finite")
    return idx[:ns[0]].astype(np.int64)


def block_select(block_scores, n_vis: int, top_k: int, C: int) -> np.ndarray:
    return _block_select(lib().oracle_block_select, block_scores, n_vis, top_k, C)


def block_select_expanded(block_scores, n_vis: int, top_k: int, C: int) -> np.ndarray:
    return _block_select(lib().oracle_block_select_expanded, block_scores, n_vis, top_k, C)


# ---------------------------------------------------------------- quantized cache

def quantize_rows(x):
    xa, xf = stored(np.asarray(x, dtype=np.float32) if not hasattr(x, "detach") else x)
    d = xa.shape[-1]
    xa = xa.reshape(-1, d)
    n = xa.shape[0]
    q8 = np.empty((n, d), np.int8)
    sc = np.empty(n, np.float32)
    lib().oracle_quantize_rows(_ptr(xa), xf, n, d, d, _ptr(q8), _ptr(sc))
    shape = np.shape(x)
    return q8.reshape(shape), sc.reshape(shape[:-1])


def dequantize_rows(q8, scale) -> np.ndarray:
    q = np.ascontiguousarray(q8, dtype=np.int8)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    d = q.shape[-1]
    out = np.empty(q.shape, np.float64)
    lib().oracle_dequantize_rows(_ptr(q), _ptr(s), q.size // d, d, _ptr(out))
    return out


# ---------------------------------------------------------------- attention

def attention_batch(q, K, V, key_off, idx, n_sel, scale: float, n_kv_heads: int = 1, dv: int | None = None):
    """Sparse attention of R query rows.

    q [R, Hq, dk]; K rows [rows, Hkv * dk] (or [rows, Hkv, dk]); V likewise
    with dv, or None for the MLA latent form (V = the first dv columns of K);
    row r attends to cache rows key_off[r] + idx[r, s] for s < n_sel[r].
    Returns float64 [R, Hq, dv]."""
    qa, qf = stored(q)
    R, Hq, dk = qa.shape
    ka, kf = stored(K)
    ka = ka.reshape(ka.shape[0], -1)
    if V is None:
        va, vf, v_stride = None, F64, 0
        dv = int(dv)
    else:
        va, vf = stored(V)
        va = va.reshape(va.shape[0], -1)
        dv = va.shape[1] // n_kv_heads
        v_stride = va.shape[1]
    ix = np.ascontiguousarray(idx, dtype=np.int32).reshape(R, -1)
    ns = np.ascontiguousarray(n_sel, dtype=np.int32)
    ko = np.ascontiguousarray(key_off, dtype=np.int64)
    out = np.empty((R, Hq, dv), np.float64)
    bad = lib().oracle_attention(R, Hq, n_kv_heads, dk, dv, _ptr(qa), qf, _ptr(ka), kf, ka.shape[1],
                                 _ptr(va) if va is not None else None, vf, v_stride, _ptr(ko), _ptr(ix),
                                 ix.shape[1], _ptr(ns), float(scale), _ptr(out))
    if bad:
        raise ValueError("negative index in a selection")
    return out


def attention_over(q, K, V, scale: float) -> np.ndarray:
    q = _f64(q)
    K = _f64(K)
    V = _f64(V)
    S = K.shape[0]
    if S == 0:
        raise ValueError("attention over an empty set")
    return attention_batch(q[None], K, V, [0], np.arange(S)[None], [S], scale)[0]


def sparse_attention_mla(q, latent, sel, scale: float, dv: int = 512) -> np.ndarray:
    sel = np.asarray(sel, dtype=np.int64)
    if sel.size == 0:
        raise ValueError("attention over an empty set")
    return attention_batch(_f64(q)[None], _f64(latent), None, [0], sel[None], [sel.size], scale, 1, dv)[0]


def sparse_attention_gqa(q, K, V, sel, scale: float) -> np.ndarray:
    K = _f64(K)
    V = _f64(V)
    sel = np.asarray(sel, dtype=np.int64)
    if sel.size == 0:
        raise ValueError("attention over an empty set")
    hkv = K.shape[1]
    return attention_batch(_f64(q)[None], K.reshape(K.shape[0], -1), V.reshape(V.shape[0], -1), [0], sel[None],
                           [sel.size], scale, hkv)[0]


def dense_attention_gqa(q, K, V, n_vis: int, scale: float) -> np.ndarray:
    return sparse_attention_gqa(q, K, V, np.arange(n_vis), scale)


def dense_attention_mla(q, latent, n_vis: int, scale: float, dv: int = 512) -> np.ndarray:
    return sparse_attention_mla(q, latent, np.arange(n_vis), scale, dv)


def decode_pipeline_mla(q_idx, w, k_cache, n_kv, top_k, q_attn, latent, scale, dv=512):
    s = indexer_scores(q_idx, w, np.asarray(k_cache)[:n_kv])
    sel = topk_select(s, n_kv, top_k)
    out = sparse_attention_mla(q_attn, latent, sel, scale, dv)
    return s, sel, out


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "ctypes", "math", "np")]
