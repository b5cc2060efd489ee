"""CPU-side tests of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every function include/lidx.h declares, and rejects bad
arguments on the host before anything is launched."""

import ctypes
import os
import re

import pytest

import lightning_indexer_top_gb300 as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    L.build()
    return L.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "lidx.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:idx_status|size_t|int32_t|const char\*)\s+(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("idx_score", "idx_score_q8", "idx_quantize_rows", "idx_block_pool", "idx_block_pool_update", "idx_topk", "sparse_attn_decode", "sparse_attn_prefill",
              "idx_hadamard", "idx_workspace_size", "idx_last_error", "idx_device_status", "idx_score_topk",
              "sparse_decode_step", "sparse_decode_step_fused", "sparse_attn_decode_noalloc", "idx_block_score_topk"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_library_is_built_for_sm103a():
    log = open(os.path.join(ROOT, "lightning_indexer_top_gb300", "_build", "api.cu.log")).read()
    assert "arch=compute_103a,code=sm_103a" in log


def _batch(n_seq=1, T=1, max_n_kv=16):
    return L._Batch(n_seq, T, ctypes.c_void_p(16), None, max_n_kv, None, max_n_kv)


def test_host_validation_rejects_bad_arguments(lib):
    # each call fails validation before any CUDA call is made
    assert lib.idx_hadamard(ctypes.c_void_p(16), ctypes.c_void_p(16), L.IDX_BF16, 4, 100, 100, None) == L.IDX_ERR_INVALID_ARG
    assert b"d must be" in lib.idx_last_error()
    assert lib.idx_hadamard(None, None, L.IDX_BF16, 4, 128, 128, None) == L.IDX_ERR_INVALID_ARG
    assert lib.idx_hadamard(ctypes.c_void_p(16), ctypes.c_void_p(16), 7, 4, 128, 128, None) == L.IDX_ERR_INVALID_ARG
    b = _batch()
    assert lib.idx_topk(None, 16, b, 0, 0, None, 16, None, None, 0, None) == L.IDX_ERR_INVALID_ARG
    assert b"top_k" in lib.idx_last_error()
    assert lib.idx_topk(None, 16, b, 32, 0, None, 16, None, None, 0, None) == L.IDX_ERR_INVALID_ARG
    assert b"capacity" in lib.idx_last_error()
    # block mode capacity = floor(top_k/C)*C + C - 1
    assert lib.idx_topk(None, 16, b, 8, 4, None, 10, None, None, 0, None) == L.IDX_ERR_INVALID_ARG
    # a page table needs page_size >= 1 and a stride covering max_n_kv
    pg = L._Batch(1, 1, ctypes.c_void_p(16), None, 0, None, 256, ctypes.c_void_p(32), 4, 0)
    assert lib.idx_topk(None, 256, pg, 8, 0, None, 8, None, None, 0, None) == L.IDX_ERR_INVALID_ARG
    pg = L._Batch(1, 1, ctypes.c_void_p(16), None, 0, None, 256, ctypes.c_void_p(32), 3, 64)
    assert lib.idx_topk(None, 256, pg, 8, 0, None, 8, None, None, 0, None) == L.IDX_ERR_INVALID_ARG
    bad = L._Batch(-1, 1, None, None, 0, None, 0)
    assert lib.idx_score(None, 0, None, 4, 32, None, 0, 32, 0, bad, 0, None, 0, None, 0, None) == L.IDX_ERR_INVALID_ARG
    assert lib.idx_score(None, 0, None, 65, 32, None, 0, 32, 0, b, 0, None, 16, None, 0, None) == L.IDX_ERR_UNSUPPORTED
    assert lib.idx_block_pool(None, L.IDX_BF16, 128, 0, b, 0, 128, None, 16, None) == L.IDX_ERR_INVALID_ARG
    assert lib.idx_block_pool_update(None, L.IDX_BF16, 128, 0, b, None, None, 0, 128, None, 16, None) == \
        L.IDX_ERR_INVALID_ARG
    assert lib.idx_quantize_rows(None, L.IDX_BF16, 4, 0, 128, None, 128, None, None) == L.IDX_ERR_INVALID_ARG
    assert lib.idx_quantize_rows(None, L.IDX_BF16, 4, 128, 128, None, 120, None, None) == L.IDX_ERR_INVALID_ARG
    # inline scales need room for the scale after the codes
    assert lib.idx_quantize_rows(ctypes.c_void_p(16), L.IDX_BF16, 4, 128, 128, ctypes.c_void_p(256), 128, None,
                                 None) == L.IDX_ERR_INVALID_ARG
    assert lib.idx_score_q8(None, L.IDX_BF16, None, 64, 128, None, 128, None, 0, b, 2, None, 16, None, 0, None) == \
        L.IDX_ERR_UNSUPPORTED
    assert lib.sparse_attn_decode(None, L.IDX_BF16, 6, 4, 128, 128, None, None, 512, 512, 0, b, None, 16, None,
                                  1.0, None, L.IDX_F32, None, 0, None) == L.IDX_ERR_INVALID_ARG
    assert b"Hq % Hkv" in lib.idx_last_error() or b"Hq" in lib.idx_last_error()
    # latent form requires one kv head
    assert lib.sparse_attn_decode(None, L.IDX_BF16, 8, 2, 576, 512, None, None, 1152, 0, 0, b, None, 16, None,
                                  1.0, None, L.IDX_F32, None, 0, None) == L.IDX_ERR_INVALID_ARG
    assert lib.sparse_attn_decode(None, L.IDX_BF16, 8, 1, 576, 512, None, None, 576, 0, 0, b, None, 16, None,
                                  float("nan"), None, L.IDX_F32, None, 0, None) == L.IDX_ERR_INVALID_ARG


def test_block_score_topk_host_validation(lib):
    # the one-call block indexer reports the three calls' argument errors, found on the host before any
    # launch: block_size < 1 and a pooled stride below max_n_kv / C (the pool's checks, made first)
    b = _batch()
    args = dict(q=None, q_dtype=L.IDX_BF16, w=None, H=32, d=128, k=None, k_dtype=L.IDX_BF16, ks=128, kr=0, b=b,
                n_pooled=None, stale=None, C=64, pooled=None, ps=16, top_k=2048, scores=None, ss=16, idx=None,
                istride=2048 + 63, n_sel=None, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.idx_block_score_topk(a["q"], a["q_dtype"], a["w"], a["H"], a["d"], a["k"], a["k_dtype"], a["ks"],
                                        a["kr"], a["b"], a["n_pooled"], a["stale"], a["C"], a["pooled"], a["ps"],
                                        a["top_k"], a["scores"], a["ss"], a["idx"], a["istride"], a["n_sel"],
                                        a["stream"])
    assert call(C=0) == L.IDX_ERR_INVALID_ARG
    assert b"block_size" in lib.idx_last_error()
    wide = L._Batch(1, 1, ctypes.c_void_p(16), None, 4096, None, 4096)
    assert call(b=wide, ps=8) == L.IDX_ERR_INVALID_ARG
    assert b"pool_seq_stride" in lib.idx_last_error()
    assert call(k_dtype=7) == L.IDX_ERR_INVALID_ARG
    # an empty batch is a no-op
    assert call(b=L._Batch(0, 1, None, None, 0, None, 0)) == L.IDX_OK


def test_empty_batch_is_a_no_op(lib):
    empty = L._Batch(0, 1, None, None, 0, None, 0)
    assert lib.idx_topk(None, 0, empty, 4, 0, None, 4, None, None, 0, None) == L.IDX_OK
    assert lib.sparse_attn_decode(None, L.IDX_BF16, 8, 1, 576, 512, None, None, 576, 0, 0, empty, None, 16,
                                  None, 1.0, None, L.IDX_F32, None, 0, None) == L.IDX_OK


def test_workspace_size_is_pure_host(lib):
    assert lib.idx_workspace_size(99, -5, -1, 0, 0, 0) == 0


def test_default_top_k_minus_one(lib):
    # -1 is the model's configured indexer top_k (2048) for sizing as for selection
    for rows in (8, 64, 1000):
        assert lib.idx_workspace_size(L.IDX_OP_TOPK, rows, 131072, -1, 0, 0) == \
            lib.idx_workspace_size(L.IDX_OP_TOPK, rows, 131072, 2048, 0, 0)
    assert L.topk_capacity(-1) == 2048


def test_mla_attention_workspace_follows_the_split_policy(lib):
    # Host policy of the MLA attention (no GPU needed; without one the library assumes GB300's 152 SMs):
    # few rows spread their selection over key splits until the 76 two-CTA clusters are covered (at least
    # 256 keys per split); a split never holds more than 2048 selected keys; one split needs no workspace,
    # otherwise every (row, split) keeps 128 heads x (512 + 2) f32 partials.
    def expected(rows, cap):
        clusters = 152 // 2
        min_s = -(-cap // 2048) if cap > 2048 else 1
        s = min(clusters // rows, -(-cap // 256)) if rows < clusters else 1
        s = max(s, min_s, 1)
        return 0 if s <= 1 else rows * s * 128 * 514 * 4
    for rows, cap in ((64, 2048), (8, 2048), (1, 2048), (75, 2048), (76, 2048), (1000, 2048), (100, 4096),
                      (8, 4096), (1, 100000), (300, 6000), (3, 300)):
        got = lib.idx_workspace_size(L.IDX_OP_ATTN_DECODE, rows, 131072, cap, 128, 512)
        assert got == expected(rows, cap), (rows, cap, got)
        assert lib.idx_workspace_size(L.IDX_OP_ATTN_PREFILL, rows, 131072, cap, 128, 512) == got
    # the headline (64 rows x 2048) needs none; 8 rows split 8 ways
    assert lib.idx_workspace_size(L.IDX_OP_ATTN_DECODE, 64, 131072, 2048, 128, 512) == 0
    assert lib.idx_workspace_size(L.IDX_OP_ATTN_DECODE, 8, 8192, 2048, 128, 512) == 8 * 8 * 128 * 514 * 4


def _step(lib, b, *, top_k=8, idx_stride=8, score_stride=16, out_dtype=L.IDX_BF16, hq=128, hkv=1, dk=576,
          dv=512, kv_stride=576, ptr=16, scale=1.0):
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.sparse_decode_step(p, L.IDX_BF16, p, 64, 128, p, L.IDX_F16, 128, 16, b, top_k, p, score_stride, p,
                                  idx_stride, p, p, L.IDX_BF16, hq, hkv, dk, dv, p, None, kv_stride, 0, 16,
                                  scale, p, out_dtype, None, 0, None)


def test_decode_step_host_validation(lib):
    # every rejection happens on the host, before anything is launched
    b = _batch()
    assert _step(lib, b, top_k=0) == L.IDX_ERR_INVALID_ARG
    assert b"top_k" in lib.idx_last_error()
    assert _step(lib, b, idx_stride=4) == L.IDX_ERR_INVALID_ARG
    assert b"idx_row_stride" in lib.idx_last_error()
    assert _step(lib, b, score_stride=8) == L.IDX_ERR_INVALID_ARG
    assert b"score_row_stride" in lib.idx_last_error()
    assert _step(lib, b, out_dtype=L.IDX_F16) == L.IDX_ERR_INVALID_ARG
    assert _step(lib, b, hq=6, hkv=4) == L.IDX_ERR_INVALID_ARG
    assert _step(lib, b, hkv=2) == L.IDX_ERR_INVALID_ARG          # latent form needs one kv head
    assert _step(lib, b, kv_stride=512) == L.IDX_ERR_INVALID_ARG
    assert b"kv_row_stride" in lib.idx_last_error()
    assert _step(lib, b, scale=float("inf")) == L.IDX_ERR_INVALID_ARG
    assert _step(lib, b, ptr=0) == L.IDX_ERR_INVALID_ARG
    assert b"NULL" in lib.idx_last_error()
    assert _step(lib, L._Batch(0, 1, None, None, 0, None, 0), ptr=0) == L.IDX_OK
    assert _step(lib, L._Batch(-1, 1, None, None, 0, None, 0)) == L.IDX_ERR_INVALID_ARG


def test_decode_step_workspace_covers_both_calls(lib):
    # the step's workspace serves the indexer's fused select and then the attention's key splits
    for rows, n_kv in ((8, 8192), (64, 131072), (1, 4096), (300, 65536)):
        a = lib.idx_workspace_size(L.IDX_OP_SCORE_TOPK, rows, n_kv, 2048, 0, 0)
        b = lib.idx_workspace_size(L.IDX_OP_ATTN_DECODE, rows, n_kv, 2048, 128, 512)
        got = lib.idx_workspace_size(L.IDX_OP_DECODE_STEP, rows, n_kv, 2048, 128, 512)
        assert got >= max(a, b)
        if rows <= 32:   # the one-launch step also keeps each row's 2048-bin score histogram
            assert got >= (-(-b // 16) * 16) + rows * 2048 * 4


def test_decode_step_fused_plan_is_host_only(lib):
    # only one query row per sequence, at most 32 rows, at most 16384 keys, and an index row that holds top_k
    assert lib.sparse_decode_step_fused(8, 2, 8192, 2048, 2048) == 0
    assert lib.sparse_decode_step_fused(33, 1, 8192, 2048, 2048) == 0
    assert lib.sparse_decode_step_fused(8, 1, 16385, 2048, 2048) == 0
    assert lib.sparse_decode_step_fused(8, 1, 8192, 2048, 1024) == 0
    assert lib.sparse_decode_step_fused(8, 1, 0, 2048, 2048) == 0
    assert lib.sparse_decode_step_fused(8, 1, 8192, 2048, 2048) in (0, 1)   # 0 without a device
