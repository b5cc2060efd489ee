"""sparse_attn_decode_noalloc: the MLA decode attention for callers that cannot
allocate device memory (its key-split scratch is a static array inside the
library).  Checked through the C ABI against sparse_attn_decode, the entry
point that takes a caller-allocated workspace, on two calls in a row: the
second call must not be disturbed by what the first left in the shared
array.  This file is collected last on purpose."""

import ctypes
import math

import pytest
import torch

import lightning_indexer_top_gb300 as L


def _case(seed, B, n_kv, sizes):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, 128, 576, generator=g).to(torch.bfloat16).cuda()
    lat = torch.randn(B * n_kv, 576, generator=g).to(torch.bfloat16).cuda()
    idx = torch.full((B, 2048), -1, dtype=torch.int32)
    for r, ns in enumerate(sizes):
        idx[r, :ns] = torch.randperm(n_kv, generator=g)[:ns].to(torch.int32)
    batch = L.Batch(torch.tensor([n_kv] * B, dtype=torch.int32, device="cuda"), 1, n_kv, kv_seq_stride=n_kv)
    return q, lat, idx.cuda(), torch.tensor(sizes, dtype=torch.int32, device="cuda"), batch


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    L.build()
    lib = L.load()
    scale = 1 / math.sqrt(192)
    cases = [(95, 8, 8192, [2048] * 8), (96, 5, 3000, [2048, 1, 700, 1999, 64])]
    for call, (seed, B, n_kv, sizes) in enumerate(cases):
        q, lat, idx, n_sel, batch = _case(seed, B, n_kv, sizes)
        # both cases split the keys of each row, so the static scratch is used
        assert L.idx_workspace_size(L.IDX_OP_ATTN_DECODE, B, n_kv, idx.shape[1], 128, 512) > 0
        ref = L.sparse_attn_decode(q, lat, None, batch, idx, n_sel, scale, dv=512, out_dtype=torch.bfloat16)
        out = torch.full((B, 128, 512), float("nan"), device="cuda", dtype=torch.bfloat16)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.sparse_attn_decode_noalloc(
            ctypes.c_void_p(q.data_ptr()), L.IDX_BF16, 128, 1, 576, 512, ctypes.c_void_p(lat.data_ptr()),
            lat.stride(0), lat.shape[0], batch.c(), ctypes.c_void_p(idx.data_ptr()), idx.stride(0),
            ctypes.c_void_p(n_sel.data_ptr()), ctypes.c_float(scale), ctypes.c_void_p(out.data_ptr()),
            L.IDX_BF16, stream)
        assert st == L.IDX_OK, lib.idx_last_error()
        torch.cuda.synchronize()
        # the same kernels with the same key splits run on both paths, only
        # the scratch memory differs: the outputs must be identical bit for bit
        assert torch.equal(out, ref), (call, (out.float() - ref.float()).abs().max().item())
    assert L.idx_device_status(reset=True) == 0


def _call_dummy(lib, n_rows, heads=128, kv_row_stride=576, idx_row_stride=16):
    # placeholder addresses: every case below is rejected on the host before any launch
    b = L._Batch(n_rows, 1, ctypes.c_void_p(16), None, 16, None, 16)
    return lib.sparse_attn_decode_noalloc(ctypes.c_void_p(16), L.IDX_BF16, heads, 1, 576, 512,
                                          ctypes.c_void_p(16), kv_row_stride, 16, b, ctypes.c_void_p(16),
                                          idx_row_stride, ctypes.c_void_p(16), ctypes.c_float(1.0),
                                          ctypes.c_void_p(16), L.IDX_BF16, None)


def test_noalloc_rejects_unsupported_shapes_without_launching():
    lib = L.load()
    assert _call_dummy(lib, 1, heads=64) == L.IDX_ERR_UNSUPPORTED
    assert b"128 query" in lib.idx_last_error()


@pytest.mark.parametrize("stride", [8, -8, 0, 575])
def test_noalloc_rejects_overlapping_latent_rows(stride):
    # rows closer than one 576-wide latent row (or running backwards) would make
    # the gather read past the caller's buffer; the workspace entry point
    # rejects them too
    lib = L.load()
    assert _call_dummy(lib, 1, kv_row_stride=stride) == L.IDX_ERR_INVALID_ARG
    assert b"kv_row_stride" in lib.idx_last_error()


def test_noalloc_rejects_calls_larger_than_the_static_array():
    # 40 rows of 4096 selected keys need two key splits each: 80 partial units,
    # more than the 76 the array holds
    lib = L.load()
    assert _call_dummy(lib, 40, idx_row_stride=4096) == L.IDX_ERR_INVALID_ARG
    assert b"static scratch array" in lib.idx_last_error()
