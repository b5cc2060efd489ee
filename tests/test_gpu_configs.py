"""End-to-end parity on the five synthetic configurations and the headline
decode workload: the whole path (Hadamard -> score -> select -> attend) runs
on the GPU exactly as the bench launches it; the C++ oracle recomputes every
row (configuration 3: rows 0-2100, which include every exactly dense row, and
every 16th row after them) from the same inputs, read as stored.

A GPU selection that differs from the oracle's by a legal near-tie swap is a
valid result too; its attention output is then checked against the oracle's
attention over that same (validated) selection.  Reports the identical-set
rate and the mean Jaccard of the selections (the pages' comparison metric)."""

import math

import numpy as np
import pytest
import torch

import oracle as O
import oracle.cpp as C
import lightning_indexer_top_gb300 as L
from lightning_indexer_top_gb300 import workloads
from lightning_indexer_top_gb300.pipeline import SparseAttentionStep
from _helpers import assert_scores_close, check_selection, np64, sorted_unique

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.build()
    L.load()
    L.idx_device_status(reset=True)
    yield
    torch.cuda.empty_cache()


def _run(wl):
    step = SparseAttentionStep(wl)
    step.run()
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    return step


def _report(name, ident):
    rate = float(np.mean([i for i, _ in ident]))
    jac = float(np.mean([j for _, j in ident]))
    print(f"\n[{name}] identical-set rate {rate:.4f}  mean Jaccard {jac:.6f}  over {len(ident)} rows")
    return rate


def _seq_arrays(wl, t, seqs):
    """Host copy of cache `t` in its storage type, and the cache row of position 0 of each sequence.
    Paged caches are gathered into position order, one sequence after another."""
    if wl.page_table is None:
        return t.cpu(), {b: wl.row0(b) for b in seqs}
    parts, off, pos = [], {}, 0
    for b in seqs:
        rows = wl.rows_of(b, wl.n_kv_host[b]).to(t.device)
        parts.append(t[rows].cpu())
        off[b] = pos
        pos += wl.n_kv_host[b]
    return torch.cat(parts), off


def _check_mla_rows(wl, step, rows, rotate=False):
    """Check rows of an MLA workload (decode or causal prefill) against the C++ oracle: scores
    (1e-3 rule), selections (identical or legal near-tie swaps), attention (2e-2 max-abs, bf16 out)."""
    rows = [int(r) for r in rows]
    seqs = sorted({r // wl.T for r in rows})
    keys, koff = _seq_arrays(wl, wl.k_idx, seqs)
    lat, loff = _seq_arrays(wl, wl.k_attn, seqs)
    sel_rows = torch.as_tensor(rows)
    q = wl.q_idx.cpu()[sel_rows]
    if rotate:
        # the cache holds rotated keys; q is rotated on its way in (both rounded once to bf16)
        keys = C.hadamard_rotate(np64(keys), store="bf16")
        q = C.hadamard_rotate(np64(q), store="bf16")
    n_vis = [C.visible_count(wl.n_kv_host[r // wl.T], None if wl.q_pos is None else r % wl.T) for r in rows]
    s_ref = C.scores_batch(q, np64(wl.w.cpu()[sel_rows]), keys, [koff[r // wl.T] for r in rows], n_vis)
    idx_ref, ns_ref = C.topk_batch(s_ref, n_vis, wl.top_k)
    s_gpu = step.scores.cpu()[sel_rows].numpy()
    idx_gpu = step.idx.cpu()[sel_rows].numpy()
    ns_gpu = step.n_sel.cpu()[sel_rows].numpy()
    ident, attend = [], np.full((len(rows), wl.top_k), -1, np.int64)
    for i, r in enumerate(rows):
        nv = n_vis[i]
        assert_scores_close(s_gpu[i, :nv], s_ref[i, :nv], f"{wl.name} row {r}")
        ns = int(ns_gpu[i])
        sel_gpu = sorted_unique(idx_gpu[i], ns)
        assert np.all(idx_gpu[i, ns:] == -1)
        sel_ref = idx_ref[i, :ns_ref[i]].tolist()
        same, jac = check_selection(sel_gpu, sel_ref, s_ref[i, :nv], f"{wl.name} row {r}")
        ident.append((same, jac))
        # the oracle attends over its own selection, or over the GPU's once it is shown to be legal
        chosen = sel_ref if same else sel_gpu
        attend[i, :len(chosen)] = chosen
    ref = C.attention_batch(wl.q_attn.cpu()[sel_rows], lat, None, [loff[r // wl.T] for r in rows], attend,
                            ns_gpu, wl.scale, 1, dv=wl.dv)
    err = np.max(np.abs(np64(step.out.cpu()[sel_rows]) - ref), axis=(1, 2))
    assert np.all(err <= 2e-2), f"{wl.name}: attention max-abs {err.max()} at row {rows[int(err.argmax())]}"
    return ident


def test_config1_tiny_prefill_fp32_all_rows():
    wl = workloads.make(1)
    step = _run(wl)
    ident = []
    qh, wh, kh = np64(wl.q_idx), np64(wl.w), np64(wl.k_idx)
    Kh, Vh = np64(wl.k_attn), np64(wl.v_attn)
    for t in range(wl.T):
        nv = t + 1
        s_ref = O.indexer_scores(qh[t], wh[t], kh[:nv])
        assert_scores_close(step.scores[t, :nv].cpu().numpy(), s_ref, f"row {t}")
        sel_ref = O.topk_select(s_ref, nv, wl.top_k)
        ns = int(step.n_sel[t])
        sel_gpu = sorted_unique(step.idx[t].cpu().numpy(), ns)
        same, jac = check_selection(sel_gpu, sel_ref, s_ref, f"row {t}")
        ident.append((same, jac))
        if nv <= wl.top_k:
            assert sel_gpu == list(range(nv))          # exactly dense below the budget
            dense = O.dense_attention_gqa(np64(wl.q_attn[t]), Kh, Vh, nv, wl.scale)
            assert np.max(np.abs(np64(step.out[t]) - dense)) <= 1e-4
        # the oracle's own selection, or the GPU's once it is shown to be a legal near-tie swap
        ref = O.sparse_attention_gqa(np64(wl.q_attn[t]), Kh, Vh, sel_ref if same else sel_gpu, wl.scale)
        assert np.max(np.abs(np64(step.out[t]) - ref)) <= 1e-4, t
    _report(wl.name, ident)


def test_config2_decode_mla_all_rows():
    wl = workloads.make(2)
    step = _run(wl)
    _report(wl.name, _check_mla_rows(wl, step, range(wl.B)))


def test_config2_batched_equals_each_sequence_alone():
    # "n_seq=4 == n_seq=1 chunk-for-chunk" (ik_llama.cpp PR #2058): a batched call is bit-identical
    wl = workloads.make(2)
    full = _run(wl)
    for b in (0, 5):
        one = workloads.make(2)
        one.B = 1
        one.q_idx, one.w, one.q_attn = wl.q_idx[b:b + 1], wl.w[b:b + 1], wl.q_attn[b:b + 1]
        one.k_idx, one.k_attn = wl.k_idx, wl.k_attn
        one.n_kv = wl.n_kv[b:b + 1].contiguous()
        one.n_kv_host = [wl.n_kv_host[b]]
        one.kv_start = torch.tensor([b * wl.kv_seq_stride], dtype=torch.int32, device="cuda")
        one.kv_start_host = [b * wl.kv_seq_stride]
        st = _run(one)
        assert torch.equal(st.scores[0], full.scores[b])
        assert torch.equal(st.idx[0], full.idx[b])
        assert torch.equal(st.out[0], full.out[b])


def test_config3_prefill_stratified_rows():
    wl = workloads.make(3)
    step = _run(wl)
    # every row up to 2100 (all the exactly dense rows and the first ones past the budget), then every 16th
    rows = list(range(0, 2101)) + list(range(2101, wl.T, 16)) + [wl.T - 1]
    _report(wl.name, _check_mla_rows(wl, step, sorted(set(rows)), rotate=True))
    for r in range(2048):   # rows below the budget are exactly dense
        assert int(step.n_sel[r]) == r + 1


def test_prefill_chunking_over_query_rows_is_bit_identical():
    # chunked prefill scoring/selection is numerically identical to one call ("Subchunk OpenPangu DSA
    # prefill gather", ik_llama_opt log): rows are independent
    wl = workloads.make(3, n_tokens_override=6000)
    step = _run(wl)
    n = wl.T
    for a, z in ((0, 2500), (2500, 6000)):
        b = L.Batch(wl.n_kv, z - a, wl.max_n_kv, kv_seq_stride=wl.kv_seq_stride, q_pos=wl.q_pos[a:z])
        s = L.idx_score(step.q_rot[a:z], wl.w[a:z], step.k_rot, b)
        idx, ns = L.idx_topk(s, b, wl.top_k)
        out = L.sparse_attn_prefill(wl.q_attn[a:z], wl.k_attn, None, b, idx, ns, wl.scale, dv=wl.dv,
                                    out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        for r in range(z - a):
            nv = a + r + 1
            assert torch.equal(s[r, :nv], step.scores[a + r, :nv])
        assert torch.equal(idx, step.idx[a:z])
        assert torch.equal(out, step.out[a:z])
    assert n == 6000


def test_config4_block_decode_all_rows_with_tails():
    wl = workloads.make(4, parity_tails=True)
    step = _run(wl)
    C = wl.block_size
    ident = []
    kh = np64(wl.k_idx)
    Kh, Vh = wl.k_attn, wl.v_attn
    for b in range(wl.B):
        n = wl.n_kv_host[b]
        row0 = wl.row0(b)
        pooled = O.block_pool(kh[row0:row0 + n], C, n)
        np.testing.assert_allclose(step.pooled[b, :n // C].cpu().numpy(), pooled, rtol=1e-5, atol=1e-6)
        bs_ref = O.indexer_scores(np64(wl.q_idx[b]), np64(wl.w[b]), pooled)
        assert_scores_close(step.scores[b, :n // C].cpu().numpy(), bs_ref, f"seq {b}")
        sel_ref = O.block_select(bs_ref, n, wl.top_k, C)
        assert np.array_equal(sel_ref, O.block_select_expanded(bs_ref, n, wl.top_k, C))
        ns = int(step.n_sel[b])
        sel_gpu = sorted_unique(step.idx[b].cpu().numpy(), ns)
        n_cb = n // C
        tail = list(range(n_cb * C, n))
        assert sel_gpu[len(sel_gpu) - len(tail):] == tail          # the tail is always kept
        gb = sorted(set(t // C for t in sel_gpu if t < n_cb * C))
        rb = sorted(set(t // C for t in sel_ref if t < n_cb * C))
        assert len([t for t in sel_gpu if t < n_cb * C]) == len(gb) * C      # whole blocks
        same, jac = check_selection(gb, rb, bs_ref, f"seq {b}")
        ident.append((same, jac))
        ref = O.sparse_attention_gqa(np64(wl.q_attn[b]), np64(Kh[row0:row0 + n]), np64(Vh[row0:row0 + n]),
                                     sel_ref if same else sel_gpu, wl.scale)
        assert np.max(np.abs(np64(step.out[b]) - ref)) <= 2e-2, b
    _report(wl.name, ident)


def test_config4_dense_threshold():
    # exactly dense at n_vis = top_k + C - 1; one more token and a block is dropped
    wl = workloads.make(4, batch_override=2, n_kv_override=2048 + 63)
    wl.n_kv = torch.tensor([2048 + 63, 2048 + 64], dtype=torch.int32, device="cuda")
    wl.n_kv_host = [2048 + 63, 2048 + 64]
    wl.max_n_kv = 2048 + 64
    wl.kv_seq_stride = 2048 + 64
    wl.k_idx = torch.randn(2 * (2048 + 64), 128, device="cuda").to(torch.bfloat16)
    wl.k_attn = torch.randn(2 * (2048 + 64), 4, 128, device="cuda").to(torch.bfloat16)
    wl.v_attn = torch.randn(2 * (2048 + 64), 4, 128, device="cuda").to(torch.bfloat16)
    step = _run(wl)
    assert int(step.n_sel[0]) == 2048 + 63
    assert step.idx[0, :2048 + 63].tolist() == list(range(2048 + 63))
    assert int(step.n_sel[1]) == 2048
    dense = O.dense_attention_gqa(np64(wl.q_attn[0]), np64(wl.k_attn[:2111]), np64(wl.v_attn[:2111]), 2111, wl.scale)
    assert np.max(np.abs(np64(step.out[0]) - dense)) <= 2e-2


def test_config5_long_ragged_decode_all_rows():
    wl = workloads.make(5)
    step = _run(wl)
    _report(wl.name, _check_mla_rows(wl, step, range(wl.B)))


def test_headline_decode_64x131072_all_rows():
    wl = workloads.make("headline")
    step = _run(wl)
    _report(wl.name, _check_mla_rows(wl, step, range(wl.B)))


def test_paged_decode_workload_all_rows():
    # the headline geometry at 8192 keys with both caches in shuffled 64-row pages
    wl = workloads.make("headline", n_kv_override=8192, batch_override=6, page_size=64)
    assert wl.page_table is not None and wl.name.endswith("_paged")
    st = _run(wl)
    _report("paged", _check_mla_rows(wl, st, range(wl.B)))


@pytest.mark.parametrize("make_args", [(("headline",), {"batch_override": 16, "n_kv_override": 65536}), ((2,), {})],
                         ids=["16x65536", "8x8192"])
def test_decode_chain_back_to_back_equals_synchronised_steps(make_args):
    # The decode kernels chain with programmatic dependent launch: each kernel may start while its
    # predecessor drains and must wait for it before touching its outputs. Alternating two query sets
    # makes any read of a stale buffer visible: back-to-back steps, never synchronised, must give exactly
    # the selections and outputs of steps synchronised after every call.
    args, kw = make_args
    wl = workloads.make(*args, **kw)
    st = SparseAttentionStep(wl)
    sets = {
        "a": (wl.q_idx.clone(), wl.w.clone(), wl.q_attn.clone()),
        "b": (wl.q_idx.flip(0).clone(), wl.w.flip(0).clone(), wl.q_attn.flip(0).clone()),
    }

    def load(name):
        q, w, qa = sets[name]
        wl.q_idx.copy_(q)
        wl.w.copy_(w)
        wl.q_attn.copy_(qa)

    ref = {}
    for name in "ab":
        load(name)
        torch.cuda.synchronize()
        for call in (st.score, st.select, st.attend):
            call()
            torch.cuda.synchronize()
        ref[name] = (st.n_sel.clone(), st.idx.clone(), st.out.clone())
    assert not torch.equal(ref["a"][1], ref["b"][1])
    got = []
    for i in range(6):
        name = "ab"[i % 2]
        load(name)
        st.run()
        got.append((name, st.n_sel.clone(), st.idx.clone(), st.out.clone()))
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    for name, n_sel, idx, out in got:
        assert torch.equal(n_sel, ref[name][0]) and torch.equal(idx, ref[name][1]), name
        assert torch.equal(out, ref[name][2]), name


@pytest.mark.parametrize("fused", [True, False], ids=["fused_select", "separate_select"])
def test_first_step_reads_the_selection_it_waits_for(fused):
    # A fresh step whose selection buffers hold sentinels: the attention, launched while the select
    # may still run (programmatic dependent launch), must read the selection that select writes,
    # not the sentinels: the step's output equals attention re-run after a full synchronisation.
    wl = workloads.make(5, batch_override=16)
    for _ in range(3):
        st = SparseAttentionStep(wl, fused=fused)
        st.idx.fill_(-7)
        st.n_sel.fill_(-7)
        st.out.zero_()
        torch.cuda.synchronize()
        st.run()
        torch.cuda.synchronize()
        first = st.out.clone()
        st.attend()
        torch.cuda.synchronize()
        assert torch.equal(first, st.out)
    assert L.idx_device_status(reset=True) == 0
