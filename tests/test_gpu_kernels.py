"""Per-kernel parity: each CUDA entry point against the CPU oracle on the same
seeded inputs, at sizes that span several tiles plus a ragged tail."""

import math

import numpy as np
import pytest
import torch

import oracle as O
import lightning_indexer_top_gb300 as L
from _helpers import assert_scores_close, np64

pytestmark = pytest.mark.gpu

DEV = "cuda"
FMT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.build()
    L.load()
    L.idx_device_status(reset=True)
    yield
    assert L.idx_device_status(reset=True) == 0


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device=DEV)


# ------------------------------------------------------------------ Hadamard

_STORE_BITS = {torch.float32: (24, -126), torch.float16: (11, -14), torch.bfloat16: (8, -126)}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
def test_hadamard_matches_oracle(dtype, d):
    # The stored rotation is the exact rotation rounded once: bit-exact against the oracle for 16-bit
    # storage.  For f32 storage the kernel's f64 rotation can, in rare near-midpoint cases, round
    # differently from the oracle's own f64 sum, so it is held to half an f32 ulp of the exact value
    # (plus the f64 error) and must agree on all but a tiny fraction of elements.
    g = torch.Generator(device=DEV).manual_seed(11 + d)
    x = torch.randn(1003, d, generator=g, device=DEV).to(dtype)
    x[0] = 0
    x[1, ::3] = 1e-3    # many equal magnitudes: exact ties at the rounding midpoints for d = 64, 256
    y = L.idx_hadamard(x, torch.empty_like(x))
    xh, got = np64(x), np64(y)
    ref = O.hadamard_rotate(xh, store=FMT[dtype])
    if dtype != torch.float32:
        np.testing.assert_array_equal(got, ref)
    else:
        exact = O.hadamard_rotate(xh)
        p, emin = _STORE_BITS[dtype]
        ulp = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(exact), 1e-300))), emin) - (p - 1))
        assert np.all(np.abs(got - exact) <= 0.5 * ulp + 1e-12 * np.abs(xh).sum(axis=1, keepdims=True))
        agree = float(np.mean(got == ref))
        print(f"\n[hadamard f32 d={d}] equal to the exact rotation rounded once: {agree:.6f}")
        assert agree > 0.9999
    # in place gives the same bits
    x2 = x.clone()
    L.idx_hadamard(x2)
    assert torch.equal(x2, y)


# ------------------------------------------------------------------ score (CUDA-core scorer)

@pytest.mark.parametrize("H,d,qt,kt", [(4, 32, torch.float32, torch.float32), (3, 40, torch.bfloat16, torch.float32),
                                       (32, 128, torch.bfloat16, torch.float32), (8, 64, torch.float16, torch.bfloat16)])
def test_score_generic_matches_oracle(H, d, qt, kt):
    g = torch.Generator(device=DEV).manual_seed(21 + H)
    B, T = 3, 5
    n_kv = [300, 129, 1]
    max_n = 300
    starts = [7, 400, 1000]
    rows = 1024
    q = torch.randn(B * T, H, d, generator=g, device=DEV).to(qt)
    w = torch.randn(B * T, H, generator=g, device=DEV) / math.sqrt(H)
    k = torch.randn(rows, d, generator=g, device=DEV).to(kt)
    q_pos = _i32([p for n in n_kv for p in (n - 1, 0, n // 2, n + 5, -1)])
    batch = L.Batch(_i32(n_kv), T, max_n, kv_start=_i32(starts), q_pos=q_pos)
    s = torch.full((B * T, max_n), 12345.0, device=DEV)
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    qh, wh, kh, sh, qp = np64(q), np64(w), np64(k), s.cpu().numpy(), q_pos.cpu().numpy()
    for r in range(B * T):
        b = r // T
        nv = O.visible_count(n_kv[b], int(qp[r]))
        ref = O.indexer_scores(qh[r], wh[r], kh[starts[b]:starts[b] + nv])
        assert_scores_close(sh[r, :nv], ref, f"row {r}")
        assert np.all(sh[r, nv:] == 12345.0), "entries past the visible keys must be untouched"


@pytest.mark.parametrize("H", [8, 16, 32, 64])
def test_score_block_mode_counts_complete_blocks(H):
    # H >= 16 takes the split-head pooled-key scorer, H = 8 the one-key-per-thread scorer
    g = torch.Generator(device=DEV).manual_seed(31 + H)
    C, d = 4, 128
    n_kv = [37, 4, 3, 64]
    B = len(n_kv)
    stride = 16
    pooled = torch.randn(B * stride, d, generator=g, device=DEV)
    if H == 32:   # more blocks than one 64-key tile of the split scorer
        n_kv = [37, 4, 3, 64 * 4 * 3 + 9]
        stride = 200
        pooled = torch.randn(B * stride, d, generator=g, device=DEV)
    q = torch.randn(B, H, d, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, H, generator=g, device=DEV)
    batch = L.Batch(_i32(n_kv), 1, max(n_kv), kv_seq_stride=stride)
    s = torch.full((B, stride), -7.0, device=DEV)
    L.idx_score(q, w, pooled, batch, block_size=C, scores=s)
    torch.cuda.synchronize()
    for b, n in enumerate(n_kv):
        nb = n // C
        ref = O.indexer_scores(np64(q[b]), np64(w[b]), np64(pooled[b * stride:b * stride + nb]))
        assert_scores_close(s[b, :nb].cpu().numpy(), ref, f"seq {b}")
        assert torch.all(s[b, nb:] == -7.0)


# ------------------------------------------------------------------ top-k (bit-exact: same f32 scores on both sides)

def _scores_cases():
    g = torch.Generator().manual_seed(41)
    yield "ties_small_ints", torch.randint(-3, 4, (6, 5000), generator=g).float()
    yield "normal", torch.randn(6, 5000, generator=g)
    yield "constant", torch.zeros(3, 3000)
    z = torch.randint(0, 2, (3, 4000), generator=g).float()
    z[z == 0] = -0.0
    z[:, ::7] = 0.0
    yield "signed_zero_ties", z
    yield "one_long_row", torch.randn(1, 131072, generator=g) * 8 + 3
    x = torch.randn(2, 70000, generator=g)
    x[:, 1000:1100] = x.max() + 1.0  # exact ties straddling the threshold
    yield "tie_block_at_top", x
    # more keys in the threshold bin than the candidate list holds
    yield "mass_ties", torch.randint(0, 2, (2, 30000), generator=g).float()
    yield "long_row_beyond_bitmap", torch.randn(1, 300000, generator=g)


def _topk_ws(path):
    # "multi": the binding sizes the workspace (several CTAs per row for few rows);
    # "single": a workspace too small for that, so one CTA handles each row
    return None if path == "multi" else torch.empty(16, device=DEV, dtype=torch.uint8)


@pytest.mark.parametrize("path", ["multi", "single"])
@pytest.mark.parametrize("case", [c for c, _ in _scores_cases()])
@pytest.mark.parametrize("top_k", [1, 64, 2048])
def test_topk_bit_exact(case, top_k, path):
    scores = dict(_scores_cases())[case]
    rows, n = scores.shape
    n_kv = [n - 37 * r for r in range(rows)]
    s = scores.to(DEV)
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=0)
    idx, n_sel = L.idx_topk(s, batch, top_k, workspace=_topk_ws(path))
    torch.cuda.synchronize()
    idx_h, ns_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    for r in range(rows):
        ref = O.topk_select(scores[r].numpy(), n_kv[r], top_k)
        assert ns_h[r] == len(ref)
        assert idx_h[r, :len(ref)].tolist() == ref.tolist(), f"row {r}"
        assert np.all(idx_h[r, len(ref):] == -1)


def _fused_case(name):
    """(q bf16 [B,64,128], w f32 [B,64], F16 key cache, n_kv per row, top_k) for the fused score + top-k."""
    g = torch.Generator().manual_seed(91)
    if name == "ragged":
        n_kv = [65536, 3000, 2048, 2049, 0, 1, 40000, 131072]
    elif name == "short_rows":
        n_kv = [8192] * 8
    elif name == "short_ragged":
        n_kv = [16384, 5000, 2048, 2049, 0, 1, 9000, 12000]
    elif name == "flat":      # one key row everywhere: every score of a row ties, the lowest positions win
        n_kv = [40000, 131072, 2049]
    else:   # "ties": every key row repeated 4 times, so each score appears 4 times (ties across the cut)
        n_kv = [20000, 65536, 4096]
    B, n = len(n_kv), max(n_kv)
    q = torch.randn(B, 64, 128, generator=g).to(torch.bfloat16)
    w = torch.randn(B, 64, generator=g) / 8
    k = torch.randn(B * n, 128, generator=g).to(torch.float16)
    if name == "flat":
        k = k[:1].expand(B * n, 128).contiguous()
    if name == "ties":
        k = k.view(B, n, 128)[:, : n // 4].unsqueeze(2).expand(B, n // 4, 4, 128).reshape(B * n, 128).contiguous()
    return q, w, k, n_kv, 2048


@pytest.mark.parametrize("name", ["ragged", "short_rows", "short_ragged", "ties", "flat"])
def test_fused_score_topk_equals_score_then_topk(name):
    # the histogram-driven select gives exactly what idx_score + idx_topk give, and what the
    # oracle's stable selection gives on the same f32 scores
    q, w, k, n_kv, top_k = _fused_case(name)
    B, n = len(n_kv), max(n_kv)
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=n)
    qd, wd, kd = q.to(DEV), w.to(DEV), k.to(DEV)
    assert L.idx_workspace_size(L.IDX_OP_SCORE_TOPK, B, n, top_k) > 0
    s1, idx1, ns1 = L.idx_score_topk(qd, wd, kd, batch, top_k)
    s2 = L.idx_score(qd, wd, kd, batch)
    idx2, ns2 = L.idx_topk(s2, batch, top_k)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    for r in range(B):
        assert torch.equal(s1[r, :n_kv[r]], s2[r, :n_kv[r]]), r
    assert torch.equal(ns1, ns2) and torch.equal(idx1, idx2)
    sh = s1.cpu().numpy()
    for r in range(B):
        ref = O.topk_select(sh[r], n_kv[r], top_k)
        assert int(ns1[r]) == len(ref) and idx1[r, :len(ref)].tolist() == ref.tolist(), r
    if name == "flat":
        for r in range(B):
            assert idx1[r, :top_k].tolist() == list(range(top_k)), r


def test_fused_score_topk_back_to_back_launches():
    # each fused launch zeroes its own histograms: repeated calls on alternating inputs give the
    # same selections as isolated calls
    q, w, k, n_kv, top_k = _fused_case("ragged")
    B, n = len(n_kv), max(n_kv)
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=n)
    qd, wd, kd = q.to(DEV), w.to(DEV), k.to(DEV)
    q2 = qd.flip(0).contiguous()
    ws = torch.empty(L.idx_workspace_size(L.IDX_OP_SCORE_TOPK, B, n, top_k), device=DEV, dtype=torch.uint8)
    ref = [L.idx_score_topk(x, wd, kd, batch, top_k, workspace=ws)[1].clone() for x in (qd, q2)]
    torch.cuda.synchronize()
    outs = [L.idx_score_topk(x, wd, kd, batch, top_k, workspace=ws)[1].clone() for x in (qd, q2, qd, q2, qd)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, ref[i % 2]), i
    assert L.idx_device_status(reset=True) == 0


@pytest.mark.parametrize("top_k", [1, 700, 2048])
def test_topk_many_short_rows_bit_exact(top_k):
    # >= 2 rows per SM and <= 16384 keys per row: the one-CTA-per-row kernel of the causal prefill.
    # Rows mix ties (small integers, signed zeros, one constant row), normal scores, ragged lengths
    # from 0 to 16384 (both sides of 9216, where the kernel loads a second batch) and dense rows.
    g = torch.Generator().manual_seed(47)
    rows, n = 320, 16384
    scores = torch.randn(rows, n, generator=g)
    scores[0::5] = torch.randint(-3, 4, (len(range(0, rows, 5)), n), generator=g).float()
    z = torch.randint(0, 2, (len(range(1, rows, 7)), n), generator=g).float()
    z[z == 0] = -0.0
    scores[1::7] = z
    scores[2] = 0.0
    n_kv = [(n - 53 * r) % (n + 1) for r in range(rows)]
    n_kv[3], n_kv[4], n_kv[5], n_kv[6] = 0, 1, top_k, top_k + 1
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=0)
    idx, n_sel = L.idx_topk(scores.to(DEV), batch, top_k)
    torch.cuda.synchronize()
    idx_h, ns_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    for r in range(rows):
        ref = O.topk_select(scores[r].numpy(), n_kv[r], top_k)
        assert ns_h[r] == len(ref), f"row {r}"
        assert idx_h[r, :len(ref)].tolist() == ref.tolist(), f"row {r}"
        assert np.all(idx_h[r, len(ref):] == -1), f"row {r}"


def test_topk_default_minus_one_equals_2048():
    g = torch.Generator().manual_seed(45)
    scores = torch.randn(3, 40000, generator=g).to(DEV)
    batch = L.Batch(_i32([40000, 3000, 1000]), 1, 40000, kv_seq_stride=0)
    a, na = L.idx_topk(scores, batch, -1)
    b, nb = L.idx_topk(scores, batch, 2048)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(na, nb)


def test_topk_multi_cta_path_with_rows_shorter_than_a_sample_block():
    # the few-long-rows path is chosen by max_n_kv; single rows in it may be tiny (n < 128)
    g = torch.Generator().manual_seed(44)
    n_kv = [40000, 100, 20, 129, 3]
    n = max(n_kv)
    scores = torch.randint(-4, 5, (len(n_kv), n), generator=g).float()
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=0)
    for top_k in (5, 64):
        idx, n_sel = L.idx_topk(scores.to(DEV), batch, top_k)
        torch.cuda.synchronize()
        for r, nv in enumerate(n_kv):
            ref = O.topk_select(scores[r].numpy(), nv, top_k)
            assert int(n_sel[r]) == len(ref) and idx[r, :len(ref)].tolist() == ref.tolist(), (top_k, r)


@pytest.mark.parametrize("path", ["multi", "single"])
def test_topk_causal_rows_and_dense_short_rows(path):
    g = torch.Generator().manual_seed(42)
    T, n, top_k = 300, 3000, 100
    scores = torch.randint(-5, 6, (T, n), generator=g).float()
    q_pos = [int(x) for x in torch.randint(-2, n + 3, (T,), generator=g)]
    batch = L.Batch(_i32([n]), T, n, kv_seq_stride=0, q_pos=_i32(q_pos))
    idx, n_sel = L.idx_topk(scores.to(DEV), batch, top_k, workspace=_topk_ws(path))
    idx_h, ns_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    for t in range(T):
        nv = O.visible_count(n, q_pos[t])
        ref = O.topk_select(scores[t].numpy(), nv, top_k)
        assert ns_h[t] == len(ref) and idx_h[t, :len(ref)].tolist() == ref.tolist(), t


@pytest.mark.parametrize("C,top_k", [(64, 2048), (4, 10), (3, 2), (8, 8)])
@pytest.mark.parametrize("many_blocks", [False, True], ids=["rank_select", "radix_select"])
def test_topk_block_mode_bit_exact(C, top_k, many_blocks):
    # rows of at most 1024 complete blocks take the rank-based select, longer ones the radix select
    g = torch.Generator().manual_seed(43 + C)
    n_vis = [top_k + C - 1, top_k + C, 0, 1, C - 1, 5 * top_k + 3, 40 * C + 17, 2 * C]
    if many_blocks:
        n_vis.append(1100 * C + 5)
    B = len(n_vis)
    nb_max = max(n_vis) // C + 1
    bscores = torch.randint(-2, 3, (B, nb_max), generator=g).float()
    batch = L.Batch(_i32(n_vis), 1, max(n_vis), kv_seq_stride=0)
    idx, n_sel = L.idx_topk(bscores.to(DEV), batch, top_k, block_size=C)
    idx_h, ns_h = idx.cpu().numpy(), n_sel.cpu().numpy()
    cap = L.topk_capacity(top_k, C)
    assert idx_h.shape[1] == cap
    for b, nv in enumerate(n_vis):
        ref = O.block_select(bscores[b].numpy(), nv, top_k, C)
        assert ns_h[b] == len(ref), b
        assert idx_h[b, :len(ref)].tolist() == ref.tolist(), b
        assert np.all(idx_h[b, len(ref):] == -1)


# ------------------------------------------------------------------ block pool

@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 64), (torch.float32, 128)])
def test_block_pool_matches_oracle(dtype, d):
    g = torch.Generator(device=DEV).manual_seed(51)
    C = 64
    n_kv = [32768 - 4 * s for s in range(3)] + [63, 64, 0]
    B = len(n_kv)
    stride_rows = 32768
    k = torch.randn(B * stride_rows, d, generator=g, device=DEV).to(dtype)
    batch = L.Batch(_i32(n_kv), 1, 32768, kv_seq_stride=stride_rows)
    pooled = L.idx_block_pool(k, batch, C, pool_seq_stride=512)
    torch.cuda.synchronize()
    kh = np64(k)
    for b, n in enumerate(n_kv):
        ref = O.block_pool(kh[b * stride_rows:b * stride_rows + n], C, n)
        got = pooled[b, :n // C].cpu().numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)


def test_block_pool_update_repools_only_new_and_stale_blocks():
    # persistent pooled cache over three "decode steps": append, edit + append, nothing new
    g = torch.Generator(device=DEV).manual_seed(52)
    C, d, stride_rows, B = 64, 128, 8192, 5
    k = torch.randn(B * stride_rows, d, generator=g, device=DEV).to(torch.bfloat16)
    n0 = [4000, 64, 0, 8191, 130]
    batch0 = L.Batch(_i32(n0), 1, 8191, kv_seq_stride=stride_rows)
    pooled = torch.full((B, 128, d), 7.0, device=DEV)
    L.idx_block_pool(k, batch0, C, pooled=pooled, pool_seq_stride=128)
    # step: sequences grow; sequence 0 edits its keys from position 1000 on, sequence 4 from 0
    n1 = [4100, 200, 63, 8191, 300]
    stale = [1000, L.IDX_POS_CLEAN, L.IDX_POS_CLEAN, L.IDX_POS_CLEAN, -1]
    k[0 * stride_rows + 1000:0 * stride_rows + 4100] = torch.randn(3100, d, generator=g, device=DEV).to(k.dtype)
    k[4 * stride_rows:4 * stride_rows + 300] = torch.randn(300, d, generator=g, device=DEV).to(k.dtype)
    before = pooled.clone()
    batch1 = L.Batch(_i32(n1), 1, 8191, kv_seq_stride=stride_rows)
    L.idx_block_pool_update(k, batch1, C, pooled, n_pooled=_i32([n // C for n in n0]), stale_pos=_i32(stale))
    torch.cuda.synchronize()
    kh, got, prev = np64(k), pooled.cpu().numpy(), before.cpu().numpy()
    for b in range(B):
        ref = O.block_pool_update(prev[b], kh[b * stride_rows:b * stride_rows + n1[b]], C, n1[b], n0[b] // C,
                                  None if stale[b] == L.IDX_POS_CLEAN else stale[b])
        nb = n1[b] // C
        np.testing.assert_allclose(got[b, :nb], ref[:nb], rtol=1e-5, atol=1e-6)
        beta0 = min(n0[b] // C, nb if stale[b] == L.IDX_POS_CLEAN else max(stale[b], 0) // C)
        assert np.array_equal(got[b, :beta0], prev[b, :beta0]), b       # untouched bits
        assert np.array_equal(got[b, nb:], prev[b, nb:]), b
    # nothing new and nothing stale: a no-op
    again = pooled.clone()
    L.idx_block_pool_update(k, batch1, C, pooled, n_pooled=_i32([n // C for n in n1]))
    torch.cuda.synchronize()
    assert torch.equal(again, pooled)


# ------------------------------------------------------------------ attention over generator-drawn index sets

def _random_sel(g, n_kv, sizes, rows):
    idx = torch.full((rows, max(sizes)), -1, dtype=torch.int32)
    for r in range(rows):
        perm = torch.randperm(n_kv, generator=g)[:sizes[r]]     # unsorted on purpose
        idx[r, :sizes[r]] = perm.to(torch.int32)
    return idx


@pytest.mark.parametrize("dtype,out_dtype", [(torch.bfloat16, torch.bfloat16), (torch.bfloat16, torch.float32),
                                             (torch.float32, torch.float32)])
def test_attention_gqa_matches_oracle(dtype, out_dtype):
    g = torch.Generator().manual_seed(61)
    B, Hq, Hkv, dh, n_kv = 5, 32, 4, 128, 3000
    sizes = [1, 31, 33, 2048, 2111]
    q = torch.randn(B, Hq, dh, generator=g).to(dtype)
    K = torch.randn(B * n_kv, Hkv, dh, generator=g).to(dtype)
    V = torch.randn(B * n_kv, Hkv, dh, generator=g).to(dtype)
    idx = _random_sel(g, n_kv, sizes, B)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    out = L.sparse_attn_decode(q.to(DEV), K.to(DEV), V.to(DEV), batch, idx.to(DEV), _i32(sizes), 1 / math.sqrt(dh),
                               out_dtype=out_dtype)
    got = np64(out)
    tol = 1e-4 if (dtype == torch.float32 and out_dtype == torch.float32) else 2e-2
    Kh, Vh = np64(K), np64(V)
    for r in range(B):
        sel = idx[r, :sizes[r]].numpy()
        ref = O.sparse_attention_gqa(np64(q[r]), Kh[r * n_kv:(r + 1) * n_kv], Vh[r * n_kv:(r + 1) * n_kv], sel,
                                     1 / math.sqrt(dh))
        assert np.max(np.abs(got[r] - ref)) <= tol, r


def test_attention_gqa_key_splits_and_fallback_without_workspace():
    # few rows: the selected keys are split over CTAs and merged (tensor cores, P rounded to bf16 for
    # the PV product: the bf16 rule); with too small a workspace for the splits the call runs one split
    # per row on the CUDA cores (f32 throughout: 1e-4); both agree with the oracle
    g = torch.Generator().manual_seed(63)
    B, Hq, Hkv, dh, n_kv = 4, 32, 4, 128, 5000
    sizes = [2111, 700, 129, 0]
    q = torch.randn(B, Hq, dh, generator=g).to(torch.bfloat16)
    K = torch.randn(B * n_kv, Hkv, dh, generator=g).to(torch.bfloat16)
    V = torch.randn(B * n_kv, Hkv, dh, generator=g).to(torch.bfloat16)
    idx = _random_sel(g, n_kv, sizes, B)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    need = L.idx_workspace_size(L.IDX_OP_ATTN_DECODE, B, n_kv, idx.shape[1], Hq, dh)
    assert need > 0
    args = (q.to(DEV), K.to(DEV), V.to(DEV), batch, idx.to(DEV), _i32(sizes), 1 / math.sqrt(dh))
    split = L.sparse_attn_decode(*args, out_dtype=torch.float32)
    single = L.sparse_attn_decode(*args, out_dtype=torch.float32,
                                  workspace=torch.empty(16, device=DEV, dtype=torch.uint8))
    torch.cuda.synchronize()
    Kh, Vh = np64(K), np64(V)
    for r in range(B):
        if sizes[r] == 0:
            assert torch.all(split[r] == 0) and torch.all(single[r] == 0)
            continue
        ref = O.sparse_attention_gqa(np64(q[r]), Kh[r * n_kv:(r + 1) * n_kv], Vh[r * n_kv:(r + 1) * n_kv],
                                     idx[r, :sizes[r]].numpy(), 1 / math.sqrt(dh))
        assert np.max(np.abs(np64(split[r]) - ref)) <= 2e-2, r
        assert np.max(np.abs(np64(single[r]) - ref)) <= 1e-4, r


@pytest.mark.parametrize("dtype,G,B", [(torch.bfloat16, 8, 16), (torch.float16, 8, 3), (torch.bfloat16, 16, 2),
                                       (torch.float16, 1, 2)])
def test_attention_gqa_tensor_cores_block_selections(dtype, G, B):
    # the block-pooled decode's shape: selections of whole 64-key blocks plus a ragged tail, dk = dv = 128,
    # G query heads per kv head; rows with an empty selection, one key, a dense row and an invalid index
    g = torch.Generator().manual_seed(64 + G)
    Hkv, dh, n_kv, C = 4, 128, 6000, 64
    Hq = G * Hkv
    q = torch.randn(B, Hq, dh, generator=g).to(dtype)
    K = torch.randn(B * n_kv, Hkv, dh, generator=g).to(dtype)
    V = torch.randn(B * n_kv, Hkv, dh, generator=g).to(dtype)
    cap = 2048 + C - 1
    idx = torch.full((B, cap), -1, dtype=torch.int32)
    sizes = []
    for r in range(B):
        kind = r % 4
        if kind == 0:      # 32 random whole blocks and the tail of the sequence
            blocks = torch.randperm(n_kv // C, generator=g)[:32].sort().values
            sel = torch.cat([(blocks[:, None] * C + torch.arange(C)).reshape(-1), torch.arange(n_kv - 37, n_kv)])
        elif kind == 1:    # one key
            sel = torch.tensor([int(torch.randint(n_kv, (1,), generator=g))])
        elif kind == 2:    # every key of a short prefix (dense)
            sel = torch.arange(700)
        else:              # nothing
            sel = torch.tensor([], dtype=torch.int64)
        idx[r, :len(sel)] = sel.to(torch.int32)
        sizes.append(len(sel))
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    args = (q.to(DEV), K.to(DEV), V.to(DEV), batch, idx.to(DEV), _i32(sizes), 1 / math.sqrt(dh))
    for out_dtype in (torch.bfloat16, torch.float32):
        out = L.sparse_attn_decode(*args, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert L.idx_device_status(reset=True) == 0
        Kh, Vh = np64(K), np64(V)
        for r in range(B):
            if sizes[r] == 0:
                assert torch.all(out[r] == 0)
                continue
            ref = O.sparse_attention_gqa(np64(q[r]), Kh[r * n_kv:(r + 1) * n_kv], Vh[r * n_kv:(r + 1) * n_kv],
                                         idx[r, :sizes[r]].numpy(), 1 / math.sqrt(dh))
            assert np.max(np.abs(np64(out[r]) - ref)) <= 2e-2, (r, out_dtype)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_attention_mla_matches_oracle(out_dtype):
    g = torch.Generator().manual_seed(62)
    B, Hq, dk, dv, n_kv = 3, 128, 576, 512, 4096
    sizes = [2048, 1, 700]
    q = torch.randn(B, Hq, dk, generator=g).to(torch.bfloat16)
    lat = torch.randn(B * n_kv, dk, generator=g).to(torch.bfloat16)
    idx = _random_sel(g, n_kv, sizes, B)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    scale = 1 / math.sqrt(192)
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale,
                               out_dtype=out_dtype, dv=dv)
    got = np64(out)
    lh = np64(lat)
    for r in range(B):
        ref = O.sparse_attention_mla(np64(q[r]), lh[r * n_kv:(r + 1) * n_kv], idx[r, :sizes[r]].numpy(), scale, dv)
        assert np.max(np.abs(got[r] - ref)) <= 2e-2, r


def test_attention_empty_selection_gives_zeros_and_bad_index_is_flagged():
    B, Hq, dh, n_kv = 2, 4, 32, 64
    q = torch.randn(B, Hq, dh, device=DEV)
    K = torch.randn(B * n_kv, 1, dh, device=DEV)
    V = torch.randn(B * n_kv, 1, dh, device=DEV)
    idx = _i32([[3, 5, 7], [1, 999, 2]])              # 999 is outside sequence 1
    n_sel = _i32([0, 3])
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    assert L.idx_device_status(reset=True) == 0
    out = L.sparse_attn_decode(q, K, V, batch, idx, n_sel, 0.5)
    assert L.idx_device_status(reset=True) == L.IDX_ERR_DEVICE_BOUNDS
    assert torch.all(out[0] == 0)
    ref = O.sparse_attention_gqa(np64(q[1]), np64(K[n_kv:]), np64(V[n_kv:]), [1, 2], 0.5)
    assert np.max(np.abs(np64(out[1]) - ref)) <= 1e-4


# ------------------------------------------------------------------ score (tensor-core decode scorer: H=64, d=128)

@pytest.mark.parametrize("qt,kt", [(torch.bfloat16, torch.float16), (torch.float16, torch.bfloat16),
                                   (torch.float32, torch.float16)])
def test_score_tensor_core_decode_matches_oracle(qt, kt):
    g = torch.Generator(device=DEV).manual_seed(71)
    n_kv = [0, 1, 129, 8192, 300, 128, 5000]
    starts = [0, 3, 100, 500, 9000, 9400, 9600]
    B, H, d, rows = len(n_kv), 64, 128, 14700
    q = torch.randn(B, H, d, generator=g, device=DEV).to(qt)
    w = torch.randn(B, H, generator=g, device=DEV) / 8
    k = torch.randn(rows, d, generator=g, device=DEV).to(kt)
    batch = L.Batch(_i32(n_kv), 1, 8192, kv_start=_i32(starts))
    s = torch.full((B, 8192), 777.0, device=DEV)
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    sh, kh = s.cpu().numpy(), np64(k)
    for b, n in enumerate(n_kv):
        ref = O.indexer_scores(np64(q[b]), np64(w[b]), kh[starts[b]:starts[b] + n])
        assert_scores_close(sh[b, :n], ref, f"seq {b}")
        assert np.all(sh[b, n:] == 777.0)


def test_score_q_beyond_f16_range_is_flagged_and_f32_q_stays_exact():
    # bf16 q against F16 keys runs on the tensor cores with q staged as f16: exact inside f16's
    # range; an element beyond it (here 1e5 -> 99840 in bf16) cannot be staged and is flagged
    g = torch.Generator(device=DEV).manual_seed(77)
    n = 4096
    q = torch.randn(2, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(2, 64, generator=g, device=DEV) / 8
    k = torch.randn(2 * n, 128, generator=g, device=DEV).to(torch.float16)
    batch = L.Batch(_i32([n, n]), 1, n, kv_seq_stride=n)
    assert L.idx_device_status(reset=True) == 0
    s = L.idx_score(q, w, k, batch)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    assert_scores_close(s[0].cpu().numpy(), O.indexer_scores(np64(q[0]), np64(w[0]), np64(k[:n])), "in range")
    q[1, 3, 7] = 1e5
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == L.IDX_ERR_INEXACT
    # f32 q of wide dynamic range (1e-8 .. 1e6 scales per head): the CUDA-core path keeps it in f32
    scale = torch.logspace(-8, 6, 64, device=DEV)[None, :, None]
    q32 = torch.randn(2, 64, 128, generator=g, device=DEV) * scale
    s32 = L.idx_score(q32, w, k, batch)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    for r in range(2):
        assert_scores_close(s32[r].cpu().numpy(), O.indexer_scores(np64(q32[r]), np64(w[r]), np64(k[r * n:(r + 1) * n])),
                            f"f32 row {r}")


def test_score_tensor_core_one_short_row_many_idle_ctas():
    # far fewer tiles than SMs: most CTAs get an empty share
    g = torch.Generator(device=DEV).manual_seed(72)
    q = torch.randn(1, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(1, 64, generator=g, device=DEV)
    k = torch.randn(300, 128, generator=g, device=DEV).to(torch.float16)
    batch = L.Batch(_i32([300]), 1, 300, kv_seq_stride=0)
    s = L.idx_score(q, w, k, batch)
    ref = O.indexer_scores(np64(q[0]), np64(w[0]), np64(k))
    assert_scores_close(s[0].cpu().numpy(), ref)


@pytest.mark.parametrize("B", [2047, 2500])
def test_score_tensor_core_decode_many_rows(B):
    # more rows than the scheduler's shared-memory prefix holds (2500: one chunk per row)
    # and just under it (2047: chunks of 8 tiles); ragged n_kv with empty rows, one shared cache
    g = torch.Generator(device=DEV).manual_seed(76)
    gc = torch.Generator().manual_seed(77)
    n_kv = torch.randint(0, 3000, (B,), generator=gc)
    n_kv[::97] = 0
    n_kv[5] = 2048 + 1
    max_n = int(n_kv.max())
    q = torch.randn(B, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, 64, generator=g, device=DEV) / 8
    k = torch.randn(max_n, 128, generator=g, device=DEV).to(torch.float16)
    batch = L.Batch(_i32(n_kv.tolist()), 1, max_n, kv_seq_stride=0)
    s = torch.full((B, max_n), 321.0, device=DEV)
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    kh = np64(k)
    for b in [0, 1, 5, 97, 1000, B - 2, B - 1] + list(range(3, B, 211)):
        n = int(n_kv[b])
        got = s[b].cpu().numpy()
        if n:
            ref = O.indexer_scores(np64(q[b]), np64(w[b]), kh[:n])
            assert_scores_close(got[:n], ref, f"row {b}")
        assert np.all(got[n:] == 321.0), b


def test_score_tensor_core_decode_back_to_back_launches():
    # the chunk counter of each launch returns to zero: many launches in a row give identical scores
    g = torch.Generator(device=DEV).manual_seed(78)
    B, n = 16, 20000
    q = torch.randn(B, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, 64, generator=g, device=DEV) / 8
    k = torch.randn(B * n, 128, generator=g, device=DEV).to(torch.float16)
    batch = L.Batch(_i32([n] * B), 1, n, kv_seq_stride=n)
    first = L.idx_score(q, w, k, batch).clone()
    for _ in range(1100):
        s = L.idx_score(q, w, k, batch)
    torch.cuda.synchronize()
    assert torch.equal(first, s)
    ref = O.indexer_scores(np64(q[3]), np64(w[3]), np64(k[3 * n:4 * n]))
    assert_scores_close(first[3].cpu().numpy(), ref)


# ------------------------------------------------------------------ MLA attention on the tensor cores

def _mla_case(seed, B, n_kv, sizes, q_scale=1.0, sorted_sel=False):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, 128, 576, generator=g) * q_scale).to(torch.bfloat16)
    lat = torch.randn(B * n_kv, 576, generator=g).to(torch.bfloat16)
    idx = _random_sel(g, n_kv, [max(s, 1) for s in sizes], B)
    if sorted_sel:
        idx = torch.sort(torch.where(idx < 0, torch.iinfo(torch.int32).max, idx), dim=1).values
        idx[idx == torch.iinfo(torch.int32).max] = -1
    return q, lat, idx


def _mla_check(q, lat, idx, sizes, n_kv, out, scale, tol=2e-2):
    got, lh = np64(out), np64(lat)
    for r, ns in enumerate(sizes):
        if ns == 0:
            assert np.all(got[r] == 0)
            continue
        ref = O.sparse_attention_mla(np64(q[r]), lh[r * n_kv:(r + 1) * n_kv], idx[r, :ns].numpy(), scale, 512)
        err = np.max(np.abs(got[r] - ref))
        assert err <= tol, (r, ns, err)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_attention_mla_tc_one_split_many_rows(out_dtype):
    # >= 76 rows: one cluster per row, no key split
    B, n_kv = 80, 700
    sizes = [(37 * r) % 700 for r in range(B)]
    sizes[3], sizes[4] = 1, 64
    q, lat, idx = _mla_case(81, B, n_kv, sizes)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    scale = 1 / math.sqrt(192)
    assert L.idx_workspace_size(L.IDX_OP_ATTN_DECODE, B, n_kv, idx.shape[1], 128, 512) == 0
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale,
                               out_dtype=out_dtype, dv=512)
    torch.cuda.synchronize()
    _mla_check(q, lat, idx, sizes, n_kv, out, scale)


def test_attention_mla_tc_split_keys_and_combine():
    # few rows: each row's keys are split over several clusters and merged
    B, n_kv = 3, 5000
    sizes = [2048, 2047, 129]
    q, lat, idx = _mla_case(82, B, n_kv, sizes)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    assert L.idx_workspace_size(L.IDX_OP_ATTN_DECODE, B, n_kv, idx.shape[1], 128, 512) > 0
    scale = 1 / math.sqrt(192)
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale, dv=512,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    _mla_check(q, lat, idx, sizes, n_kv, out, scale)


def test_attention_mla_tc_growing_maxima_rescale():
    # large logits with keys visited in ascending-logit order: the running maximum
    # jumps by far more than 2^8 between tiles, exercising the O rescale path
    B, n_kv = 2, 4096
    g = torch.Generator().manual_seed(83)
    q = (torch.randn(B, 128, 576, generator=g) * 4).to(torch.bfloat16)
    lat = torch.randn(B * n_kv, 576, generator=g)
    # later positions -> larger logits, through the 64 rope columns only, so the value
    # part (first 512 columns) stays N(0, 1)
    lat[:, 512:] *= torch.linspace(0.1, 12.0, n_kv).repeat(B)[:, None]
    lat = lat.to(torch.bfloat16)
    sizes = [2048, 1500]
    idx = torch.full((B, 2048), -1, dtype=torch.int32)
    for r in range(B):
        idx[r, :sizes[r]] = torch.arange(0, 2 * sizes[r], 2, dtype=torch.int32)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    scale = 1 / math.sqrt(192)
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale, dv=512,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    _mla_check(q, lat, idx, sizes, n_kv, out, scale)


def test_attention_mla_tc_empty_rows_and_invalid_index():
    B, n_kv = 80, 300
    sizes = [0 if r % 5 == 0 else 70 for r in range(B)]
    q, lat, idx = _mla_case(84, B, n_kv, sizes)
    idx[1, 5] = 5000                                           # outside the sequence
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=n_kv)
    scale = 1 / math.sqrt(192)
    assert L.idx_device_status(reset=True) == 0
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale, dv=512,
                               out_dtype=torch.float32)
    assert L.idx_device_status(reset=True) == L.IDX_ERR_DEVICE_BOUNDS
    keep = [j for j in range(70) if j != 5]
    ref = O.sparse_attention_mla(np64(q[1]), np64(lat[n_kv:2 * n_kv]), idx[1, keep].numpy(), scale, 512)
    assert np.max(np.abs(np64(out[1]) - ref)) <= 2e-2
    rest = [r for r in range(B) if r != 1]
    _mla_check(q[rest], lat.view(B, n_kv, 576)[rest].reshape(-1, 576), idx[rest], [sizes[r] for r in rest], n_kv,
               out[rest], scale)


def test_attention_mla_tc_selections_longer_than_one_split():
    # selections above 4096 keys always split, even with many rows; all rows share one cache
    B, n_kv, cap = 80, 6000, 5000
    g = torch.Generator().manual_seed(85)
    q = torch.randn(B, 128, 576, generator=g).to(torch.bfloat16)
    lat = torch.randn(n_kv, 576, generator=g).to(torch.bfloat16)
    sizes = [cap if r % 3 == 0 else (r * 61) % cap + 1 for r in range(B)]
    idx = torch.full((B, cap), -1, dtype=torch.int32)
    for r in range(B):
        idx[r, :sizes[r]] = torch.randperm(n_kv, generator=g)[:sizes[r]].to(torch.int32)
    batch = L.Batch(_i32([n_kv] * B), 1, n_kv, kv_seq_stride=0)
    assert L.idx_workspace_size(L.IDX_OP_ATTN_DECODE, B, n_kv, cap, 128, 512) > 0
    scale = 1 / math.sqrt(192)
    out = L.sparse_attn_decode(q.to(DEV), lat.to(DEV), None, batch, idx.to(DEV), _i32(sizes), scale, dv=512,
                               out_dtype=torch.float32)
    got, lh = np64(out), np64(lat)
    for r in range(0, B, 7):
        ref = O.sparse_attention_mla(np64(q[r]), lh, idx[r, :sizes[r]].numpy(), scale, 512)
        assert np.max(np.abs(got[r] - ref)) <= 2e-2, r


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
def test_score_tensor_core_prefill_matches_oracle(dt):
    # two sequences of 300 query rows each (not a multiple of the 128-row tile), continuing
    # after cached prefixes of different lengths: q_pos = prefix + t
    g = torch.Generator(device=DEV).manual_seed(73)
    B, T, H, d = 2, 300, 64, 128
    prefix = [700, 40]
    n_kv = [p + T for p in prefix]
    max_n = max(n_kv)
    q = torch.randn(B * T, H, d, generator=g, device=DEV).to(dt)
    w = torch.randn(B * T, H, generator=g, device=DEV) / 8
    k = torch.randn(B * max_n, d, generator=g, device=DEV).to(dt)
    q_pos = _i32([p + t for p in prefix for t in range(T)])
    batch = L.Batch(_i32(n_kv), T, max_n, kv_seq_stride=max_n, q_pos=q_pos)
    s = torch.full((B * T, max_n), 555.0, device=DEV)
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    sh, kh = s.cpu().numpy(), np64(k)
    for r in [0, 1, 127, 128, 129, 255, 299, 300, 301, 450, 599]:
        b, t = divmod(r, T)
        nv = prefix[b] + t + 1
        ref = O.indexer_scores(np64(q[r]), np64(w[r]), kh[b * max_n:b * max_n + nv])
        assert_scores_close(sh[r, :nv], ref, f"row {r}")
        assert np.all(sh[r, nv:] == 555.0)


def test_score_tensor_core_prefill_many_short_sequences():
    # 4100 sequences of 64 query rows: more (sequence, query tile) pairs than one launch
    # enumerates, some sequences without keys, and query positions out of order within a
    # sequence (the visible-key bound of a tile is the largest of its rows)
    g = torch.Generator(device=DEV).manual_seed(74)
    B, T, H, d, max_n = 4100, 64, 64, 128, 300
    n_kv = [(b * 37) % (max_n + 1) for b in range(B)]
    q = torch.randn(B * T, H, d, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(B * T, H, generator=g, device=DEV) / 8
    k = torch.randn(B * max_n, d, generator=g, device=DEV).to(torch.bfloat16)
    gc = torch.Generator().manual_seed(75)
    q_pos = torch.cat([torch.randint(-1, max(n, 1), (T,), generator=gc) for n in n_kv]).to(torch.int32)
    batch = L.Batch(_i32(n_kv), T, max_n, kv_seq_stride=max_n, q_pos=q_pos.to(DEV))
    s = torch.full((B * T, max_n), 555.0, device=DEV)
    L.idx_score(q, w, k, batch, scores=s)
    torch.cuda.synchronize()
    rows = [0, 63, 64 * 37 + 5] + list(range(64 * 4095, 64 * 4100, 13)) + list(range(101, B * T, 9973))
    qp = q_pos.numpy()
    for r in rows:
        b = r // T
        nv = min(int(qp[r]) + 1, n_kv[b]) if qp[r] >= 0 else 0
        got = s[r].cpu().numpy()
        if nv:
            ref = O.indexer_scores(np64(q[r]), np64(w[r]), np64(k[b * max_n:b * max_n + nv]))
            assert_scores_close(got[:nv], ref, f"row {r}")
        assert np.all(got[nv:] == 555.0), r


# ------------------------------------------------------------------ quantized (int8 + per-row scale) key cache

@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float16, 128), (torch.float32, 40)])
def test_quantize_rows_bit_exact(dtype, d):
    g = torch.Generator(device=DEV).manual_seed(81)
    n = 3001
    x = (torch.randn(n, d, generator=g, device=DEV) * torch.rand(n, 1, generator=g, device=DEV) * 10).to(dtype)
    x[7] = 0
    x[11, :] = 127.0
    x[11, 1] = 2.5
    q8, sc = L.idx_quantize_rows(x)
    torch.cuda.synchronize()
    rq, rs = O.quantize_rows(np64(x))
    assert np.array_equal(sc.cpu().numpy(), rs)
    assert np.array_equal(q8.cpu().numpy(), rq)


def _q8_cache(g, rows, d=128):
    k = torch.randn(rows, d, generator=g, device=DEV) * torch.rand(rows, 1, generator=g, device=DEV) * 3
    return L.idx_quantize_rows(k)


@pytest.mark.parametrize("qt", [torch.bfloat16, torch.float16])
def test_score_q8_tensor_core_decode_matches_oracle(qt):
    g = torch.Generator(device=DEV).manual_seed(82)
    n_kv = [0, 1, 129, 8192, 300, 128, 5000, 20000]
    starts = [0, 3, 100, 500, 9000, 9400, 9600, 15000]
    B, H, d, rows = len(n_kv), 64, 128, 35000
    q = torch.randn(B, H, d, generator=g, device=DEV).to(qt)
    w = torch.randn(B, H, generator=g, device=DEV) / 8
    k8, ks = _q8_cache(g, rows)
    ks[9001] = -ks[9001]                     # a negative scale: relu(scale * dot) per head
    batch = L.Batch(_i32(n_kv), 1, 20000, kv_start=_i32(starts))
    s = torch.full((B, 20000), 777.0, device=DEV)
    L.idx_score_q8(q, w, k8, ks, batch, scores=s)
    torch.cuda.synchronize()
    sh = s.cpu().numpy()
    kd = O.dequantize_rows(k8.cpu().numpy(), ks.cpu().numpy())
    for b, n in enumerate(n_kv):
        ref = O.indexer_scores(np64(q[b]), np64(w[b]), kd[starts[b]:starts[b] + n])
        assert_scores_close(sh[b, :n], ref, f"seq {b}")
        assert np.all(sh[b, n:] == 777.0)


def test_score_q8_generic_path_matches_oracle():
    # 32 heads x 64 and f32 q go to the CUDA-core scorer
    g = torch.Generator(device=DEV).manual_seed(83)
    n_kv = [40, 700, 1]
    B, rows = 3, 1000
    for H, d, qt in [(32, 64, torch.bfloat16), (64, 128, torch.float32)]:
        q = torch.randn(B, H, d, generator=g, device=DEV).to(qt)
        w = torch.randn(B, H, generator=g, device=DEV) / 8
        k8, ks = _q8_cache(g, rows, d)
        batch = L.Batch(_i32(n_kv), 1, 700, kv_seq_stride=0)
        s = L.idx_score_q8(q, w, k8, ks, batch)
        torch.cuda.synchronize()
        kd = O.dequantize_rows(k8.cpu().numpy(), ks.cpu().numpy())
        for b, n in enumerate(n_kv):
            ref = O.indexer_scores(np64(q[b]), np64(w[b]), kd[:n])
            assert_scores_close(s[b, :n].cpu().numpy(), ref, f"H={H} seq {b}")


def test_score_q8_selection_matches_oracle_at_128k():
    # one row at the headline length: scores on sampled keys, then the top-2048 set
    g = torch.Generator(device=DEV).manual_seed(84)
    n = 131072
    q = torch.randn(2, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(2, 64, generator=g, device=DEV) / 8
    k8, ks = _q8_cache(g, 2 * n)
    batch = L.Batch(_i32([n, n]), 1, n, kv_seq_stride=n)
    s = L.idx_score_q8(q, w, k8, ks, batch)
    idx, ns = L.idx_topk(s, batch, 2048)
    torch.cuda.synchronize()
    kd = O.dequantize_rows(k8[n:].cpu().numpy(), ks[n:].cpu().numpy())
    ref = O.indexer_scores(np64(q[1]), np64(w[1]), kd)
    assert_scores_close(s[1].cpu().numpy(), ref, "row 1")
    from _helpers import check_selection
    check_selection(idx[1, :int(ns[1])].cpu().numpy(), O.topk_select(ref, n, 2048), ref, "q8 row 1")


# ------------------------------------------------------------------ paged caches (cell -> position maps)

def _page(g, keys_per_seq, P, spare=7):
    """Scatter per-sequence rows (lists of [n, ...] tensors) into shuffled pages of P rows.
    Returns (paged rows, page_table [B, pages] int32 CUDA)."""
    B = len(keys_per_seq)
    pages = max((k.shape[0] + P - 1) // P for k in keys_per_seq)
    n_phys = B * pages + spare
    perm = torch.randperm(n_phys, generator=g)
    table = perm[:B * pages].view(B, pages).to(torch.int32)
    shape = (n_phys * P,) + tuple(keys_per_seq[0].shape[1:])
    rows = torch.zeros(shape, dtype=keys_per_seq[0].dtype, device=DEV)
    for b, k in enumerate(keys_per_seq):
        for lp in range((k.shape[0] + P - 1) // P):
            seg = k[lp * P:(lp + 1) * P]
            ph = int(table[b, lp])
            rows[ph * P:ph * P + seg.shape[0]] = seg
    return rows, table.to(DEV)


@pytest.mark.parametrize("P", [64, 256])
def test_paged_decode_path_is_bit_identical_to_contiguous(P):
    # scores (F16 keys and int8 keys), selection and MLA attention read the same key rows
    # in the same order whichever way the cache is laid out
    g = torch.Generator().manual_seed(91)
    n_kv = [3000, 129, 64, 5000]
    B = len(n_kv)
    gd = torch.Generator(device=DEV).manual_seed(92)
    keys = [torch.randn(n, 128, generator=gd, device=DEV).to(torch.float16) for n in n_kv]
    lats = [torch.randn(n, 576, generator=gd, device=DEV).to(torch.bfloat16) for n in n_kv]
    q = torch.randn(B, 64, 128, generator=gd, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, 64, generator=gd, device=DEV) / 8
    qa = torch.randn(B, 128, 576, generator=gd, device=DEV).to(torch.bfloat16)
    starts = [0]
    for n in n_kv[:-1]:
        starts.append(starts[-1] + n)
    kc, lc = torch.cat(keys), torch.cat(lats)
    contig = L.Batch(_i32(n_kv), 1, max(n_kv), kv_start=_i32(starts))
    kp, table = _page(g, keys, P)
    lp, table2 = _page(torch.Generator().manual_seed(91), lats, P)
    assert torch.equal(table, table2)
    paged = L.Batch(_i32(n_kv), 1, max(n_kv), page_table=table, page_size=P)
    s_c = L.idx_score(q, w, kc, contig)
    s_p = L.idx_score(q, w, kp, paged)
    k8c, scc = L.idx_quantize_rows(kc)
    k8p, scp = L.idx_quantize_rows(kp)
    q8_c = L.idx_score_q8(q, w, k8c, scc, contig)
    q8_p = L.idx_score_q8(q, w, k8p, scp, paged)
    rc, _ = L.idx_quantize_rows(kc, inline_scale=True)
    rp, _ = L.idx_quantize_rows(kp, inline_scale=True)
    qi_c = L.idx_score_q8(q, w, rc, None, contig)
    qi_p = L.idx_score_q8(q, w, rp, None, paged)
    idx_c, ns_c = L.idx_topk(s_c, contig, 2048)
    idx_p, ns_p = L.idx_topk(s_p, paged, 2048)
    o_c = L.sparse_attn_decode(qa, lc, None, contig, idx_c, ns_c, 1 / math.sqrt(192), dv=512)
    o_p = L.sparse_attn_decode(qa, lp, None, paged, idx_p, ns_p, 1 / math.sqrt(192), dv=512)
    torch.cuda.synchronize()
    for b, n in enumerate(n_kv):
        assert torch.equal(s_c[b, :n], s_p[b, :n]), b
        assert torch.equal(q8_c[b, :n], q8_p[b, :n]), b
        assert torch.equal(qi_c[b, :n], qi_p[b, :n]) and torch.equal(qi_c[b, :n], q8_c[b, :n]), b
    assert torch.equal(idx_c, idx_p) and torch.equal(ns_c, ns_p)
    assert torch.equal(o_c, o_p)
    ref = O.indexer_scores(np64(q[3]), np64(w[3]), np64(keys[3]))
    assert_scores_close(s_p[3, :n_kv[3]].cpu().numpy(), ref, "paged row 3")


def test_paged_generic_paths_match_oracle():
    # page size 48 (not a multiple of 64) and 32 heads: CUDA-core scorer, pool and GQA attention
    g = torch.Generator().manual_seed(93)
    gd = torch.Generator(device=DEV).manual_seed(94)
    P, C = 48, 16
    n_kv = [700, 47, 200]
    B = len(n_kv)
    keys = [torch.randn(n, 64, generator=gd, device=DEV).to(torch.bfloat16) for n in n_kv]
    kv = [torch.randn(n, 2, 64, generator=gd, device=DEV).to(torch.bfloat16) for n in n_kv]
    vv = [torch.randn(n, 2, 64, generator=gd, device=DEV).to(torch.bfloat16) for n in n_kv]
    kp, table = _page(g, keys, P)
    Kp, _ = _page(torch.Generator().manual_seed(93), kv, P)
    Vp, _ = _page(torch.Generator().manual_seed(93), vv, P)
    paged = L.Batch(_i32(n_kv), 1, max(n_kv), page_table=table, page_size=P)
    q = torch.randn(B, 32, 64, generator=gd, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, 32, generator=gd, device=DEV) / 8
    s = L.idx_score(q, w, kp, paged)
    pooled = L.idx_block_pool(kp, paged, C)
    qa = torch.randn(B, 8, 64, generator=gd, device=DEV).to(torch.bfloat16)
    sel = torch.full((B, 64), -1, dtype=torch.int32)
    sizes = []
    for b, n in enumerate(n_kv):
        m = min(n, 64)
        sel[b, :m] = torch.randperm(n, generator=g)[:m].to(torch.int32)
        sizes.append(m)
    out = L.sparse_attn_decode(qa, Kp, Vp, paged, sel.to(DEV), _i32(sizes), 0.125, dv=64, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for b, n in enumerate(n_kv):
        ref = O.indexer_scores(np64(q[b]), np64(w[b]), np64(keys[b]))
        assert_scores_close(s[b, :n].cpu().numpy(), ref, f"seq {b}")
        np.testing.assert_allclose(pooled[b, :n // C].cpu().numpy(), O.block_pool(np64(keys[b]), C, n),
                                   rtol=1e-5, atol=1e-6)
        ro = O.sparse_attention_gqa(np64(qa[b]), np64(kv[b]), np64(vv[b]), sel[b, :sizes[b]].numpy(), 0.125)
        assert np.max(np.abs(out[b].cpu().numpy() - ro)) <= 1e-4


def test_paged_prefill_scores_match_contiguous():
    # causal prefill on the tensor cores: 64-row page pieces of the 256-key tiles
    g = torch.Generator().manual_seed(95)
    gd = torch.Generator(device=DEV).manual_seed(96)
    T, P = 700, 128
    k = torch.randn(T, 128, generator=gd, device=DEV).to(torch.bfloat16)
    q = torch.randn(T, 64, 128, generator=gd, device=DEV).to(torch.bfloat16)
    w = torch.randn(T, 64, generator=gd, device=DEV) / 8
    kp, table = _page(g, [k], P)
    qp = _i32(list(range(T)))
    contig = L.Batch(_i32([T]), T, T, kv_seq_stride=T, q_pos=qp)
    paged = L.Batch(_i32([T]), T, T, q_pos=qp, page_table=table, page_size=P)
    s_c = torch.full((T, T), 9.0, device=DEV)
    s_p = torch.full((T, T), 9.0, device=DEV)
    L.idx_score(q, w, k, contig, scores=s_c)
    L.idx_score(q, w, kp, paged, scores=s_p)
    torch.cuda.synchronize()
    assert torch.equal(s_c, s_p)


def test_quantize_and_score_with_inline_scales():
    # rows of 144 bytes: 128 codes, the f32 scale in bytes 128..131; the same codes and scales as
    # the separate layout, and scores of the dequantized keys (tensor-core and CUDA-core paths)
    g = torch.Generator(device=DEV).manual_seed(86)
    n = 9000
    k = torch.randn(n, 128, generator=g, device=DEV) * torch.rand(n, 1, generator=g, device=DEV) * 3
    rows, none = L.idx_quantize_rows(k, inline_scale=True)
    assert none is None and rows.stride(0) == 144
    k8s, scs = L.idx_quantize_rows(k)
    torch.cuda.synchronize()
    assert torch.equal(rows[:, :128], k8s) and torch.equal(L.inline_scales(rows, 128), scs)
    n_kv = [0, 1, 300, 8192, 500]
    starts = [0, 1, 10, 400, 8500]
    B = len(n_kv)
    q = torch.randn(B, 64, 128, generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn(B, 64, generator=g, device=DEV) / 8
    batch = L.Batch(_i32(n_kv), 1, 8192, kv_start=_i32(starts))
    s_in = torch.full((B, 8192), 5.0, device=DEV)
    L.idx_score_q8(q, w, rows, None, batch, scores=s_in)
    s_sep = L.idx_score_q8(q, w, k8s, scs, batch)
    qf = q.float()   # f32 q: the CUDA-core path with inline scales
    s_gen = L.idx_score_q8(qf, w, rows, None, batch)
    torch.cuda.synchronize()
    kd = O.dequantize_rows(k8s.cpu().numpy(), scs.cpu().numpy())
    for b, nk in enumerate(n_kv):
        assert torch.equal(s_in[b, :nk], s_sep[b, :nk]), b
        assert np.all(s_in[b, nk:].cpu().numpy() == 5.0)
        ref = O.indexer_scores(np64(q[b]), np64(w[b]), kd[starts[b]:starts[b] + nk])
        assert_scores_close(s_in[b, :nk].cpu().numpy(), ref, f"inline seq {b}")
        assert_scores_close(s_gen[b, :nk].cpu().numpy(), ref, f"inline generic seq {b}")


def _block_step_case(name):
    """(q, w, raw keys, n_kv, H, mode, stale) for the one-call block-pooled indexer."""
    g = torch.Generator().manual_seed(1234)
    H, kdt, mode, stale = 32, torch.bfloat16, "update", None
    n_kv = [32768 - 4 * s for s in range(16)]
    if name == "ragged_full":          # blocks of one key row short, empty rows, dense rows, a full pooling
        n_kv, mode = [20000, 63, 0, 64, 2111, 2112, 2175, 65536], "full"
    elif name == "stale_f16_64heads":  # edits re-pool from the stale block on
        H, kdt, stale = 64, torch.float16, [100, 2 ** 31 - 1, 0, 30000, 5000, -1, 64, 32767]
        n_kv = [32768, 32000, 20000, 32768, 8000, 4096, 128, 32768]
    elif name == "f32_12heads":
        H, kdt = 12, torch.float32
    elif name == "8heads_three_calls":  # below the one launch's head range: the three calls inside
        H = 8
    elif name == "rows_200":           # more rows than SMs: one CTA per row
        n_kv = [4096 - 8 * (s % 7) for s in range(200)]
    elif name == "paged_raw":          # the raw keys in shuffled pages of 64 rows
        n_kv = [5000, 32768, 64, 20000]
    B, n = len(n_kv), max(n_kv)
    q = torch.randn(B, H, 128, generator=g).to(torch.bfloat16)
    w = torch.randn(B, H, generator=g) / math.sqrt(H)
    k = torch.randn(B * n, 128, generator=g).to(kdt)
    return q, w, k, n_kv, H, mode, stale


@pytest.mark.parametrize("name", ["decode16", "ragged_full", "stale_f16_64heads", "f32_12heads",
                                  "8heads_three_calls", "rows_200", "paged_raw"])
def test_block_score_topk_equals_the_three_calls(name):
    # pool update + pooled-key score + block select in one call: the pooled cache, the block scores
    # and the selection bit for bit those of idx_block_pool_update, idx_score and idx_topk
    q, w, k, n_kv, H, mode, stale = _block_step_case(name)
    B, n, C, top_k = len(n_kv), max(n_kv), 64, 2048
    ps = n // C
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=n)
    pool_batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=ps)
    qd, wd, kd = q.to(DEV), w.to(DEV), k.to(DEV)
    if name == "paged_raw":
        kd, table = _page(torch.Generator().manual_seed(5), [kd[b * n:b * n + n_kv[b]] for b in range(B)], 64)
        batch = L.Batch(_i32(n_kv), 1, n, page_table=table, page_size=64)
    pooled0 = L.idx_block_pool(kd, batch, C, pool_seq_stride=ps)
    n_cb = [x // C for x in n_kv]
    n_pooled = stale_pos = None
    if mode == "update":
        n_pooled = _i32([max(c - 1, 0) for c in n_cb] if stale is None else n_cb)
        first = [max(c - 1, 0) for c in n_cb] if stale is None else \
            [min(c, 0 if s < 0 else s // C) for c, s in zip(n_cb, stale)]
        for b in range(B):   # what must be re-pooled holds garbage before the call
            pooled0[b, first[b]:n_cb[b]] = 1e6
        if stale is not None:
            stale_pos = _i32(stale)
    else:
        pooled0.fill_(1e6)
    pooled_ref, pooled_one = pooled0.clone(), pooled0.clone()
    L.idx_block_pool_update(kd, batch, C, pooled_ref, n_pooled=n_pooled, stale_pos=stale_pos, pool_seq_stride=ps)
    s_ref = L.idx_score(qd, wd, pooled_ref.view(-1, 128), pool_batch, block_size=C)
    i_ref, ns_ref = L.idx_topk(s_ref, batch, top_k, block_size=C)
    s_one, i_one, ns_one = L.idx_block_score_topk(qd, wd, kd, batch, C, pooled_one, top_k, n_pooled=n_pooled,
                                                  stale_pos=stale_pos, pool_seq_stride=ps)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    assert torch.equal(pooled_ref, pooled_one)
    for r in range(B):
        assert torch.equal(s_ref[r, :n_cb[r]], s_one[r, :n_cb[r]]), r
    assert torch.equal(ns_ref, ns_one) and torch.equal(i_ref, i_one)
    # and the selection is the oracle's block selection of those scores
    sh = s_one.cpu().numpy()
    for r in range(0, B, max(1, B // 8)):
        ref = O.block_select(sh[r, :n_cb[r]], n_kv[r], top_k, C)
        assert int(ns_one[r]) == len(ref) and i_one[r, :len(ref)].tolist() == list(ref), r


@pytest.mark.parametrize("planted", [0, 150])
def test_topk_long_rows_threshold_ties(planted):
    # few long rows (the multi-CTA select: sampled bound, filter, finish): the finish ranks the keys that
    # share the threshold's top 22 bits directly when they are few, and by a histogram when many are
    # equal (planted copies of the top_k-th score)
    g = torch.Generator().manual_seed(4242 + planted)
    rows, n, top_k = 4, 131072, 2048
    s = torch.randn(rows, n, generator=g)
    if planted:
        for r in range(rows):
            t = torch.sort(s[r], descending=True).values[top_k - 1]
            pos = torch.randperm(n, generator=g)[:planted]
            s[r, pos] = t
    n_kv = [n, n - 1000, n - 77, n]
    batch = L.Batch(_i32(n_kv), 1, n, kv_seq_stride=0)
    ws = torch.empty(L.idx_workspace_size(L.IDX_OP_TOPK, rows, n, top_k), device=DEV, dtype=torch.uint8)
    idx, n_sel = L.idx_topk(s.to(DEV), batch, top_k, workspace=ws)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    for r in range(rows):
        ref = O.topk_select(s[r].numpy(), n_kv[r], top_k)
        assert int(n_sel[r]) == len(ref) and idx[r, :len(ref)].cpu().tolist() == ref.tolist(), r
