"""The decode step in one launch (sparse_decode_step): for few short decode rows the library runs
scores, top-k and the MLA attention as one kernel.  Its scores, selection and output must be bit for
bit those of idx_score_topk followed by sparse_attn_decode (the two calls, themselves checked against
the oracle elsewhere), and a sample of rows is checked against the C++ oracle directly."""

import types

import numpy as np
import pytest
import torch

import lightning_indexer_top_gb300 as L
from lightning_indexer_top_gb300 import workloads
from lightning_indexer_top_gb300.pipeline import SparseAttentionStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    L.build()
    L.load()
    L.idx_device_status(reset=True)
    yield
    torch.cuda.empty_cache()


def _set_lengths(wl, lengths):
    """Shorten the sequences of a workload in place (the caches keep their rows)."""
    wl.n_kv_host = list(lengths)
    wl.n_kv.copy_(torch.tensor(lengths, dtype=torch.int32, device=wl.n_kv.device))
    return wl


def _workload(case):
    if case == "config2":
        return workloads.make(2)
    if case == "short_rows":          # 3000 keys: a ragged last tile, top_k below n_kv
        return workloads.make(2, n_kv_override=3000)
    if case == "ragged":              # dense rows (n_kv <= top_k), a row of one key, an empty row
        return _set_lengths(workloads.make(2), [8192, 2048, 2047, 2049, 1, 0, 5000, 129])
    if case == "paged":
        return workloads.make(2, page_size=64)
    if case == "one_row":
        return workloads.make(2, batch_override=1)
    if case == "rows_32":
        return workloads.make(2, batch_override=32, n_kv_override=4096)
    if case == "ties":                # all scores 0: the lowest positions win every tie
        wl = workloads.make(2, batch_override=4)
        wl.q_idx.zero_()
        return wl
    raise ValueError(case)


def _two_calls(wl, out_dtype):
    b = L.Batch(wl.n_kv, 1, wl.max_n_kv, kv_start=wl.kv_start, kv_seq_stride=wl.kv_seq_stride,
                page_table=wl.page_table, page_size=wl.page_size)
    scores, idx, n_sel = L.idx_score_topk(wl.q_idx, wl.w, wl.k_idx, b, wl.top_k)
    out = L.sparse_attn_decode(wl.q_attn, wl.k_attn, None, b, idx, n_sel, wl.scale, out_dtype=out_dtype, dv=wl.dv)
    return scores, idx, n_sel, out


def _one_call(wl, out_dtype):
    b = L.Batch(wl.n_kv, 1, wl.max_n_kv, kv_start=wl.kv_start, kv_seq_stride=wl.kv_seq_stride,
                page_table=wl.page_table, page_size=wl.page_size)
    return L.sparse_decode_step(wl.q_idx, wl.w, wl.k_idx, b, wl.top_k, wl.q_attn, wl.k_attn, None, wl.scale,
                                dv=wl.dv, out_dtype=out_dtype)


def _assert_same(a, b, wl):
    s1, i1, n1, o1 = a
    s2, i2, n2, o2 = b
    for r, nv in enumerate(wl.n_kv_host):
        assert torch.equal(s1[r, :nv], s2[r, :nv]), f"scores of row {r}"
    assert torch.equal(n1, n2)
    assert torch.equal(i1, i2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("case", ["config2", "short_rows", "ragged", "paged", "one_row", "rows_32", "ties"])
def test_decode_step_equals_the_two_calls(case):
    wl = _workload(case)
    rows = wl.B
    assert L.sparse_decode_step_fused(rows, 1, wl.max_n_kv, wl.top_k, wl.top_k), "expected one launch"
    for out_dtype in (torch.bfloat16, torch.float32):
        ref = _two_calls(wl, out_dtype)
        got = _one_call(wl, out_dtype)
        torch.cuda.synchronize()
        assert L.idx_device_status(reset=True) == 0
        _assert_same(ref, got, wl)
    if case == "ties":
        idx, n_sel = got[1], got[2]
        assert torch.equal(idx[:, :wl.top_k].cpu(), torch.arange(wl.top_k, dtype=torch.int32).expand(rows, -1))
    if case == "ragged":
        n_sel = got[2].cpu().tolist()
        assert n_sel == [min(n, wl.top_k) for n in wl.n_kv_host]
        assert torch.all(got[3][5].float() == 0)          # the empty row attends to nothing
        assert torch.all(got[1][5] == -1)


def test_decode_step_runs_as_one_kernel():
    wl = workloads.make(2)
    _one_call(wl, torch.bfloat16)
    torch.cuda.synchronize()
    prof = pytest.importorskip("torch.profiler")
    with prof.profile(activities=[prof.ProfilerActivity.CUDA]) as p:
        _one_call(wl, torch.bfloat16)
        torch.cuda.synchronize()
    names = [e.name for e in p.events() if e.device_type == prof.DeviceType.CUDA]
    lib_kernels = [n for n in names if "lidx" in n]
    if not names:
        pytest.skip("the profiler recorded no CUDA kernels here")
    assert len(lib_kernels) == 1 and "decode_fused_kernel" in lib_kernels[0], lib_kernels


def test_decode_step_back_to_back_reuses_its_sync_slots():
    # more calls than the 256 slots of flags and counters: every call must leave its slot at zero
    wl = workloads.make(2, batch_override=4, n_kv_override=4096)
    first = _one_call(wl, torch.bfloat16)
    b = L.Batch(wl.n_kv, 1, wl.max_n_kv, kv_start=wl.kv_start, kv_seq_stride=wl.kv_seq_stride)
    scores, idx, n_sel, out = (torch.empty_like(t) for t in first)
    ws = torch.empty(L.idx_workspace_size(L.IDX_OP_DECODE_STEP, wl.B, wl.max_n_kv, wl.top_k, 128, wl.dv),
                     device="cuda", dtype=torch.uint8)
    for _ in range(300):
        L.sparse_decode_step(wl.q_idx, wl.w, wl.k_idx, b, wl.top_k, wl.q_attn, wl.k_attn, None, wl.scale,
                             dv=wl.dv, scores=scores, idx=idx, n_sel=n_sel, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    _assert_same(first, (scores, idx, n_sel, out), wl)


def test_decode_step_matches_the_oracle():
    # the step as the bench runs it (pipeline in one call) against the C++ oracle on every row
    from test_gpu_configs import _check_mla_rows, _report
    wl = _set_lengths(workloads.make(2), [8192, 3000, 2048, 100, 8192, 6000, 4097, 1])
    step = SparseAttentionStep(wl)
    assert step.one_launch and step.launches_per_step() == 1
    step.run()
    torch.cuda.synchronize()
    assert L.idx_device_status(reset=True) == 0
    ident = _check_mla_rows(wl, step, range(wl.B))
    assert _report("decode step, one launch", ident) >= 0.5
