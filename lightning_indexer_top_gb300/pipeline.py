"""One pass of the hot path over a workload: (Hadamard) -> score -> select -> attend.

Buffers are allocated once at construction; ``run()`` only enqueues the
library's kernels on the current stream, so a step can be timed, repeated or
captured in a CUDA graph.  This is orchestration only: every arithmetic step
is a call into liblidx.
"""

from __future__ import annotations

import torch

from . import Batch, idx_block_pool, idx_hadamard, idx_score, idx_score_q8, idx_topk, idx_workspace_size, topk_capacity
from . import idx_block_score_topk, idx_score_topk, IDX_OP_SCORE_TOPK, sparse_decode_step, sparse_decode_step_fused, IDX_OP_DECODE_STEP
from . import sparse_attn_decode, sparse_attn_prefill, IDX_OP_ATTN_DECODE, IDX_OP_ATTN_PREFILL, IDX_OP_TOPK
from .workloads import Workload


class SparseAttentionStep:
    """pool: block-pooled workloads only.  "full" pools every complete block in every step;
    "update" keeps the pooled keys across steps (pooled once at construction) and each step
    re-pools only the newest complete block of every sequence, as a decode step does when
    its token has just completed a block (idx_block_pool_update)."""

    def __init__(self, wl: Workload, out_dtype=None, pool: str = "full", fused: bool = True,
                 one_call: bool = True):
        self.wl = wl
        self.pool_mode = pool
        dev = wl.q_idx.device
        self.batch = Batch(wl.n_kv, wl.T, wl.max_n_kv, kv_start=wl.kv_start, kv_seq_stride=wl.kv_seq_stride,
                           q_pos=wl.q_pos, page_table=wl.page_table, page_size=wl.page_size)
        rows = wl.B * wl.T
        C = wl.block_size
        if C > 1:
            self.pool_stride = max(wl.max_n_kv // C, 1)
            self.pooled = torch.zeros(wl.B, self.pool_stride, wl.d, device=dev, dtype=torch.float32)
            self.pool_batch = Batch(wl.n_kv, wl.T, wl.max_n_kv, kv_seq_stride=self.pool_stride, q_pos=wl.q_pos)
            n_keys = self.pool_stride
            if pool == "update":
                self.n_pooled = torch.clamp(wl.n_kv // C - 1, min=0).to(torch.int32).contiguous()
                idx_block_pool(wl.k_idx, self.batch, C, pool_seq_stride=self.pool_stride, pooled=self.pooled)
        else:
            n_keys = max(wl.max_n_kv, 1)
        self.scores = torch.empty(rows, n_keys, device=dev, dtype=torch.float32)
        cap = topk_capacity(wl.top_k, C)
        self.idx = torch.empty(rows, cap, device=dev, dtype=torch.int32)
        self.n_sel = torch.empty(rows, device=dev, dtype=torch.int32)
        # decode rows over token keys in a 16-bit cache: scoring and selection in one fused call
        self.fused = fused and C <= 1 and wl.k8 is None and wl.T == 1 and wl.H == 64 and wl.d == 128
        op = IDX_OP_SCORE_TOPK if self.fused else IDX_OP_TOPK
        tws = idx_workspace_size(op, rows, wl.max_n_kv, wl.top_k) if C <= 1 else 0
        self.topk_ws = torch.empty(tws, device=dev, dtype=torch.uint8) if tws else None
        if out_dtype is None:   # f32 in -> f32 out, 16-bit in -> bf16 out
            out_dtype = torch.float32 if wl.q_attn.dtype == torch.float32 else torch.bfloat16
        self.out = torch.empty(rows, wl.q_attn.shape[1], wl.dv, device=dev, dtype=out_dtype)
        op = IDX_OP_ATTN_PREFILL if wl.kind == "prefill" else IDX_OP_ATTN_DECODE
        ws = idx_workspace_size(op, rows, wl.max_n_kv, cap, wl.q_attn.shape[1], wl.dv)
        self.attn_ws = torch.empty(max(ws, 16), device=dev, dtype=torch.uint8) if ws else None
        self.attn = sparse_attn_prefill if wl.kind == "prefill" else sparse_attn_decode
        # MLA decode over few short rows: the whole step as one call (sparse_decode_step), one launch
        self.one_call = (one_call and self.fused and wl.kind == "decode" and wl.v_attn is None and
                         wl.q_attn.shape[1] == 128 and not wl.hadamard and
                         sparse_decode_step_fused(rows, wl.T, wl.max_n_kv, wl.top_k, cap))
        self.one_launch = self.one_call
        self.step_ws = None
        if self.one_call:
            sws = idx_workspace_size(IDX_OP_DECODE_STEP, rows, wl.max_n_kv, wl.top_k, 128, wl.dv)
            self.step_ws = torch.empty(sws, device=dev, dtype=torch.uint8) if sws else None
        self.q_rot = None
        self.k_rot = None
        if wl.hadamard:
            self.q_rot = torch.empty_like(wl.q_idx)
            self.k_rot = torch.empty_like(wl.k_idx)

    def rotate(self):
        """Hadamard-rotate q and k into separate buffers (the cache holds rotated keys)."""
        idx_hadamard(self.wl.q_idx, self.q_rot)
        idx_hadamard(self.wl.k_idx, self.k_rot)

    def score(self):
        wl = self.wl
        q = wl.q_idx if self.q_rot is None else self.q_rot
        k = wl.k_idx if self.k_rot is None else self.k_rot
        if wl.block_size > 1:
            # pool update (or a full pooling), pooled-key scores and block selection in one call
            n_pooled = self.n_pooled if self.pool_mode == "update" else None
            idx_block_score_topk(q, wl.w, k, self.batch, wl.block_size, self.pooled, wl.top_k, n_pooled=n_pooled,
                                 pool_seq_stride=self.pool_stride, scores=self.scores, idx=self.idx,
                                 n_sel=self.n_sel)
        elif wl.k8 is not None:
            idx_score_q8(q, wl.w, wl.k8, wl.k_scale, self.batch, scores=self.scores)
        elif self.one_call:
            sparse_decode_step(q, wl.w, k, self.batch, wl.top_k, wl.q_attn, wl.k_attn, None, wl.scale, dv=wl.dv,
                               scores=self.scores, idx=self.idx, n_sel=self.n_sel, out=self.out,
                               workspace=self.step_ws)
        elif self.fused:
            idx_score_topk(q, wl.w, k, self.batch, wl.top_k, scores=self.scores, idx=self.idx, n_sel=self.n_sel,
                           workspace=self.topk_ws)
        else:
            idx_score(q, wl.w, k, self.batch, scores=self.scores)

    def select(self):
        if self.fused or self.wl.block_size > 1:
            return   # selected by the fused call in score()
        idx_topk(self.scores, self.batch, self.wl.top_k, block_size=self.wl.block_size, idx=self.idx,
                 n_sel=self.n_sel, workspace=self.topk_ws)

    def attend(self):
        wl = self.wl
        if self.one_call:
            return   # attended by the one call in score()
        if wl.v_attn is None:
            self.attn(wl.q_attn, wl.k_attn, None, self.batch, self.idx, self.n_sel, wl.scale, out=self.out,
                      workspace=self.attn_ws, dv=wl.dv)
        else:
            self.attn(wl.q_attn, wl.k_attn, wl.v_attn, self.batch, self.idx, self.n_sel, wl.scale,
                      out=self.out, workspace=self.attn_ws)

    def run(self):
        if self.q_rot is not None:
            self.rotate()
        self.score()
        self.select()
        self.attend()
        return self.out

    def _gqa_split_pair(self) -> bool:
        """Whether the tensor-core GQA attention runs its rows' keys as two splits, which a 2-CTA
        cluster merges itself (no combine launch): the library's split rule for that kernel."""
        wl = self.wl
        if wl.v_attn is None or wl.dv != 128 or wl.q_attn.shape[2] != 128 or wl.q_attn.dtype == torch.float32:
            return False
        rows, hq, hkv = wl.B * wl.T, wl.q_attn.shape[1], wl.v_attn.shape[1]
        if hq % hkv or hq // hkv > 16:
            return False
        cap = self.idx.shape[1]
        sms = torch.cuda.get_device_properties(self.idx.device).multi_processor_count
        s = max(min(sms // max(rows * hkv, 1), -(-cap // 256)), -(-cap // 2048), 1)
        if s > 1:
            fit = (self.attn_ws.numel() if self.attn_ws is not None else 0) // (rows * hq * 130 * 4)
            s = min(s, fit) if fit > 1 else 1
        return s == 2

    def launches_per_step(self) -> int:
        """Kernels one run() enqueues (library launches only)."""
        if self.one_launch:
            return 1
        wl = self.wl
        combine = 1 if self.attn_ws is not None and not self._gqa_split_pair() else 0
        n = 3 + combine   # score, select, attend (+ split combine)
        if wl.block_size > 1:
            # pool update + pooled-key scores + block select: one launch for decode rows of 9-64 heads and
            # at most 1024 blocks, else three
            one = wl.T == 1 and 9 <= wl.H <= 64 and wl.max_n_kv // wl.block_size <= 1024
            return (1 if one else 3) + n - 2 + (2 if self.q_rot is not None else 0)
        if self.fused:
            # fused select: one kernel for rows up to 16384 keys, else bound, filter, finish
            n += 0 if self.wl.max_n_kv <= 16384 else 2
        elif self.topk_ws is not None:
            n += 2                              # multi-CTA select: bound, filter, finish
        if self.q_rot is not None:
            n += 2                              # two Hadamard rotations
        return n
