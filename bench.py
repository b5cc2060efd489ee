#!/usr/bin/env python3
"""Throughput of one decode step of lightning-indexer sparse attention.

Workload (one step): 64 decode queries, each over n_kv = 131072 cached tokens:
score every key with the 64-head x 128-dim indexer (F16 key cache), select
top_k = 2048 keys per query, and run MLA attention (128 heads, 576-wide bf16
latent, 512-wide value) over the selected keys.  Synthetic, seeded data.

Prints ONE JSON line (rank 0):
  value       queries/s, device-resident inputs, CUDA events: the median of
              repeated windows of K steps (spread reported)
  e2e         the same metric through the public API with pinned host buffers:
              per step H2D of the step's query inputs and D2H of its output
  roofline    the dominant kernel against the measured peak (HBM copy or bf16)
  configs     every other configuration timed in the same run: per-kernel
              medians, rooflines, and its parity sample against the C++ oracle
  cpu_baseline  the C++ oracle (OpenMP over query rows, all host cores) on the
              whole step's 64 queries; also the full parity record of the step

`--impl reference` times the C++ oracle instead (the reference arm).
Multi-GPU (torchrun): each rank runs its own 64-query batch (weak scaling),
no data-path collective; the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn decode queries/s at n_kv=128K,top_k=2048; key-cache GB/s vs HBM peak"
UNIT = "queries/s"
WORKLOAD = "decode_mla_64x131072"

# name -> (workloads.make arguments, SparseAttentionStep arguments); the first is the headline the
# bench line reports.  Others serve the per-configuration lines and profiling captures on smaller cases.
WORKLOADS = {
    "decode_mla_64x131072": (("headline",), {}, {}),
    "decode_mla_8x131072": (("headline",), {"batch_override": 8}, {}),
    "decode_mla_16x131072": (("headline",), {"batch_override": 16}, {}),
    "decode_mla_8x8192": ((2,), {}, {}),
    "decode_mla_64x8192": (("headline",), {"n_kv_override": 8192}, {}),
    "long_decode_mla_ragged": ((5,), {}, {}),
    "decode_mla_64x131072_q8": (("headline",), {"quantized_keys": True}, {}),
    "decode_mla_8x131072_q8": (("headline",), {"batch_override": 8, "quantized_keys": True}, {}),
    "decode_mla_64x131072_paged": (("headline",), {"page_size": 64}, {}),
    "prefill_mla_16384": ((3,), {}, {}),
    "prefill_mla_4096": ((3,), {"n_tokens_override": 4096}, {}),
    "block_decode_gqa_16x32768": ((4,), {}, {"pool": "update"}),
}
# the configurations timed beside the headline in a default run (configuration 1 is a parity case only)
CONFIG_LINES = ["decode_mla_8x8192", "prefill_mla_16384", "block_decode_gqa_16x32768", "long_decode_mla_ragged"]

# DRAM bytes of the decode scorer per key from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch over 8 rows x 131072 keys, scaled to a launch by the keys
# it scans), keyed by the SHA-256 of the kernel source it was taken on and the indexer cache (F16
# rows or int8 codes + scale).  A source change makes the figure stale and the bench reports
# traffic = null.
NCU_TRAFFIC = {
    ("be41d910d0faeb047ff57344c2b357cd8742db8d6dd9e7413861b008c6d82c37", "f16"): (268662784 + 4388352) / (8 * 131072),
    ("be41d910d0faeb047ff57344c2b357cd8742db8d6dd9e7413861b008c6d82c37", "q8"): (138649344 + 3528960) / (8 * 131072),
}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0=None, t1=None):
        """Clock summary over the samples taken between host times t0 and t1 (all if None)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, power, smax, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's value (step times are reported as the max over ranks)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world_size: int, units_per_rank: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's step time."""
    return world_size * units_per_rank / (ms_per_step * 1e-3)


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


# ------------------------------------------------------------------ timing

KERNELS = ("hadamard", "score", "topk", "attention")


def time_step(step, stream, steps: int, warmup: int, min_ms: float = 0.0, sampler=None):
    """Warm-up, then windows of `steps` steps until at least `min_ms` of timed work (one window at
    least).  Each window is bracketed by synchronisation and timed with two CUDA events on `stream`
    around its steps, which run back to back as a serving loop runs them (nothing is recorded
    between the kernels, so launches chained on the device stay chained).  One more window of
    `steps` steps with an event between consecutive calls gives the per-kernel times.  Returns the
    window step times, the per-kernel medians and the host time span of the step-time windows."""
    import torch
    rotates = step.q_rot is not None
    calls = (step.rotate if rotates else None, step.score, step.select, step.attend)
    for _ in range(max(warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    windows = []
    t_host0 = time.perf_counter()
    spent = 0.0
    while not windows or spent < min_ms:
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        w0.record(stream)
        for _ in range(steps):
            step.run()
        w1.record(stream)
        torch.cuda.synchronize()
        ms = w0.elapsed_time(w1)
        windows.append(ms / steps)
        spent += ms
    t_host1 = time.perf_counter()
    per_kernel = {k: [] for k in KERNELS}
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        for j, call in enumerate(calls):
            evs[i][j].record(stream)
            if call is not None:
                call()
        evs[i][4].record(stream)
    torch.cuda.synchronize()
    for e in evs:
        for j, k in enumerate(KERNELS):
            per_kernel[k].append(e[j].elapsed_time(e[j + 1]))
    med = {k: statistics.median(v) for k, v in per_kernel.items()}
    if not rotates:
        med["hadamard"] = 0.0
    return windows, med, (t_host0, t_host1)


# ------------------------------------------------------------------ rooflines

def rooflines(wl, step, ms, hbm, bf16, peak_kind):
    """Per-kernel rooflines (algorithmic bytes or flops per launch / median launch time) and the
    dominant kernel's.  Bytes and flops per unit:
      decode scan      key row (2d B F16, d + 4 B int8) + 4 B score per key; q (H d x 2 B) and w (H x 4 B) per row
      prefill score    2 H d flops per (row, visible key)
      block score      pooled key (4 d B) + 4 B score per complete block; q, w per row
      top-k            4 B per score read + 4 B per selected index written
      MLA attention    1152 B gathered per selected key + q (128 x 576 x 2 B) + out per row;
                       128 x (576 + 512) x 2 flops per selected key
      GQA attention    Hkv (dk + dv) x 2 B gathered per selected key + q + out per row
      block pool       C d x 2 B read + 4 d B written per re-pooled block
    """
    B = wl.B * wl.T
    C = wl.block_size
    if wl.q_pos is not None:
        n_vis = [min(t + 1, wl.n_kv_host[0]) for t in range(wl.T)] * wl.B
    else:
        n_vis = [n for n in wl.n_kv_host for _ in range(wl.T)]
    n_sel = [min(n, wl.top_k) for n in n_vis] if C <= 1 else [
        min(wl.top_k // C, n // C) * C + n % C for n in n_vis]
    out_bytes = 2
    q_bytes = wl.q_idx.element_size()
    r = {}

    def hbm_line(kernel, nbytes, t_ms):
        a = nbytes / (t_ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": a, "peak": hbm, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": a / hbm, "algorithmic_bytes_per_launch": nbytes, "ms": t_ms}

    def tensor_line(kernel, flops, t_ms):
        a = flops / (t_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": kernel, "achieved": a, "peak": bf16, "peak_kind": peak_kind,
                "unit": "TFLOP/s", "frac": a / bf16, "algorithmic_flops_per_launch": flops, "ms": t_ms}

    if getattr(step, "one_launch", False):
        # the whole step in one kernel: the scan's bytes (keys, scores, q, w), the selection written,
        # and the attention's (gathered latent rows, q, out)
        n_keys = sum(wl.n_kv_host)
        dk = wl.q_attn.shape[-1]
        nbytes = (n_keys * (wl.d * 2 + 4) + B * wl.H * (wl.d * q_bytes + 4) + sum(n_sel) * 4 +
                  sum(n_sel) * dk * 2 + B * wl.q_attn.shape[1] * (dk * 2 + wl.dv * out_bytes))
        t = ms["score"]   # the one call (select and attend are empty in this pipeline)
        r["step"] = hbm_line("sparse_decode_step (score + top-k + MLA attention, one launch)", nbytes, t)
        r["step"]["tensor_frac"] = (2.0 * n_keys * wl.H * wl.d + 2.0 * sum(n_sel) * wl.q_attn.shape[1] *
                                    (dk + wl.dv)) / (t * 1e-3) / 1e12 / bf16
        return r, "step"
    if wl.kind == "prefill":
        r["score"] = tensor_line("idx_score (prefill, tcgen05)", 2.0 * sum(n_vis) * wl.H * wl.d, ms["score"])
    elif C > 1:
        n_cb = sum(n // C for n in wl.n_kv_host)
        nbytes = n_cb * (wl.d * 4 + 4) + B * wl.H * (wl.d * q_bytes + 4)
        # the step also re-pools the newest block of every sequence and writes the selection; one call
        # (idx_block_score_topk: pool update + pooled-key scores + block select)
        nbytes += wl.B * (C * wl.d * wl.k_idx.element_size() + wl.d * 4) + sum(n_sel) * 4
        r["score"] = hbm_line("idx_block_score_topk (pool update + pooled-key scores + block select, one launch)",
                              nbytes, ms["score"] + ms["topk"])
    else:
        n_keys = sum(wl.n_kv_host)
        per_key = wl.d * 2 if wl.k8 is None else wl.d + 4
        nbytes = n_keys * (per_key + 4) + B * wl.H * (wl.d * q_bytes + 4)
        if step.fused:
            # one call: the scan (with the histogram epilogue) and the two select kernels; the bytes are
            # the scan's (keys read, scores written, q and w read) plus the selection written
            r["score"] = hbm_line("idx_score_topk (key-cache scan + histogram select)",
                                  nbytes + sum(n_sel) * 4, ms["score"] + ms["topk"])
        else:
            r["score"] = hbm_line("idx_score (key-cache scan)" if wl.k8 is None else
                                  "idx_score_q8 (int8 key-cache scan)", nbytes, ms["score"])
    n_scores = sum(n_vis) if C <= 1 else sum(n // C for n in n_vis)
    if not getattr(step, "fused", False) and C <= 1:
        r["topk"] = hbm_line("idx_topk", n_scores * 4 + sum(n_sel) * 4, ms["topk"])
    Hq, dk = wl.q_attn.shape[1], wl.q_attn.shape[-1]
    if wl.v_attn is None:
        nbytes = sum(n_sel) * dk * 2 + B * Hq * (dk * 2 + wl.dv * out_bytes)
        flops = 2.0 * sum(n_sel) * Hq * (dk + wl.dv)
        if wl.kind == "prefill":
            r["attention"] = tensor_line("sparse_attn_prefill (MLA, tcgen05)", flops, ms["attention"])
        else:
            r["attention"] = hbm_line("sparse_attn_decode (MLA, tcgen05)", nbytes, ms["attention"])
            r["attention"]["tensor_frac"] = flops / (ms["attention"] * 1e-3) / 1e12 / bf16
    else:
        Hkv = wl.k_attn.shape[1]
        nbytes = sum(n_sel) * Hkv * (dk + wl.dv) * 2 + B * Hq * (dk + wl.dv) * 2
        tc = (str(wl.k_attn.dtype) in ("torch.float16", "torch.bfloat16") and dk == 128 and wl.dv == 128
              and Hq % Hkv == 0 and Hq // Hkv <= 16)
        r["attention"] = hbm_line("sparse_attn_decode (GQA, %s)" % ("tcgen05" if tc else "CUDA cores"), nbytes,
                                  ms["attention"])
    if wl.hadamard:
        nbytes = 2 * (wl.q_idx.numel() + wl.k_idx.numel()) * wl.q_idx.element_size()
        r["hadamard"] = hbm_line("idx_hadamard (q and k)", nbytes, ms["hadamard"])
    dominant = max(r, key=lambda k: r[k]["ms"])
    return r, dominant


# ------------------------------------------------------------------ the C++ oracle on the same inputs

def oracle_parity(wl, step, rows):
    """Run the C++ oracle (score -> select -> attend) on the given query rows of a workload and compare
    with the step's results.  Returns (wall seconds of the oracle, parity record)."""
    import numpy as np
    import torch
    import oracle.cpp as C
    rows = [int(r) for r in rows]
    sel_rows = torch.as_tensor(rows)
    seqs = sorted({r // wl.T for r in rows})
    Cb = wl.block_size

    def host(t):
        if wl.page_table is None:
            return t.cpu(), {b: wl.row0(b) for b in seqs}
        parts, off, pos = [], {}, 0
        for b in seqs:
            parts.append(t[wl.rows_of(b, wl.n_kv_host[b]).to(t.device)].cpu())
            off[b] = pos
            pos += wl.n_kv_host[b]
        return torch.cat(parts), off

    keys, koff = host(wl.k_idx if wl.k8 is None else wl.k8[:, :wl.d])
    kscale = None
    if wl.k8 is not None:   # the quantized cache: codes and their per-row scales, gathered the same way
        kscale = host(wl.k_scale.view(-1, 1))[0].view(-1).numpy()
    lat, loff = host(wl.k_attn)
    vals = host(wl.v_attn)[0] if wl.v_attn is not None else None
    q = wl.q_idx.cpu()[sel_rows]
    w = wl.w.cpu()[sel_rows].double().numpy()
    qa = wl.q_attn.cpu()[sel_rows]
    n_vis = [C.visible_count(wl.n_kv_host[r // wl.T], None if wl.q_pos is None else r % wl.T) for r in rows]
    t0 = time.perf_counter()
    if wl.hadamard:
        keys = C.hadamard_rotate(keys.double().numpy(), store="bf16")
        q = C.hadamard_rotate(q.double().numpy(), store="bf16")
    if Cb > 1:
        n_cb = [n // Cb for n in n_vis]
        pooled = np.zeros((len(seqs), max(max(wl.n_kv_host) // Cb, 1), wl.d), np.float32)
        for i, b in enumerate(seqs):
            k_seq = keys[koff[b]:koff[b] + wl.n_kv_host[b]]
            pooled[i, :wl.n_kv_host[b] // Cb] = C.block_pool(k_seq, Cb, wl.n_kv_host[b])
        pooled_flat = pooled.reshape(-1, wl.d)
        boff = [seqs.index(r // wl.T) * pooled.shape[1] for r in rows]
        s_ref = C.scores_batch(q, w, pooled_flat, boff, n_cb)
        sel_ref = [C.block_select(s_ref[i], n_vis[i], wl.top_k, Cb) for i in range(len(rows))]
    else:
        s_ref = C.scores_batch(q, w, keys, [koff[r // wl.T] for r in rows], n_vis, k_scale=kscale)
        idx_ref, ns_ref = C.topk_batch(s_ref, n_vis, wl.top_k)
        sel_ref = [idx_ref[i, :ns_ref[i]] for i in range(len(rows))]
    cap = max(len(s) for s in sel_ref) if sel_ref else 1
    attend = np.full((len(rows), max(cap, 1)), -1, np.int64)
    for i, s in enumerate(sel_ref):
        attend[i, :len(s)] = s
    n_att = [len(s) for s in sel_ref]
    Hkv = 1 if wl.v_attn is None else wl.k_attn.shape[1]
    out_ref = C.attention_batch(qa, lat, vals, [loff[r // wl.T] for r in rows], attend, n_att, wl.scale, Hkv,
                                dv=wl.dv)
    dt = time.perf_counter() - t0
    # compare
    s_gpu = step.scores.cpu()[sel_rows].numpy()
    idx_gpu = step.idx.cpu()[sel_rows].numpy()
    ns_gpu = step.n_sel.cpu()[sel_rows].numpy()
    out_gpu = step.out.cpu()[sel_rows].double().numpy()
    same, jac, rel, oerr = [], [], 0.0, 0.0
    for i in range(len(rows)):
        nv = n_vis[i] if Cb <= 1 else n_vis[i] // Cb
        ref = s_ref[i, :nv].astype(np.float64)
        if nv:
            floor = 1e-2 * np.max(np.abs(ref))
            rel = max(rel, float(np.max(np.abs(s_gpu[i, :nv] - ref) / np.maximum(np.maximum(np.abs(ref), floor),
                                                                                   1e-30))))
        a = set(idx_gpu[i, :ns_gpu[i]].tolist())
        b = set(int(x) for x in sel_ref[i])
        same.append(a == b)
        jac.append(len(a & b) / len(a | b) if (a | b) else 1.0)
        if a == b:
            oerr = max(oerr, float(np.max(np.abs(out_gpu[i] - out_ref[i]))))
    rec = {"rows": len(rows), "identical_set_rate": float(np.mean(same)), "mean_jaccard": float(np.mean(jac)),
           "max_score_rel_err": rel, "max_out_abs_err_identical_rows": oerr,
           "score_tolerance": "1e-3 x max(|s|, 1e-2 max_row |s|)", "out_tolerance": "2e-2 (bf16 out)"}
    return dt, rec


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """Reference arm: the C++ oracle, as it stands, on bounded samples of the headline workload."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle.cpp as C
    from lightning_indexer_top_gb300 import workloads
    cores = C.threads()
    n = max(1, min(cores, 64))
    wl = workloads.make("headline", device="cpu", batch_override=n)

    def one_step():
        rows = list(range(n))
        s = C.scores_batch(wl.q_idx, wl.w.double().numpy(), wl.k_idx, [wl.row0(b) for b in rows], wl.n_kv_host)
        idx, ns = C.topk_batch(s, wl.n_kv_host, wl.top_k)
        C.attention_batch(wl.q_attn, wl.k_attn, None, [wl.row0(b) for b in rows], idx, ns, wl.scale, 1, dv=wl.dv)

    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        one_step()
    t = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one_step()
        t += time.perf_counter() - t0
    v = n * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs)",
            "config": {"workload": WORKLOAD, "sample": f"{n} of the 64 queries of the workload per step",
                       "top_k": 2048, "n_kv": 131072},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle (C++17, OpenMP over rows)",
                             "sample": f"{n} decode queries (n_kv=131072) per step: score, top-k, MLA attention"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ native arm

def make_step(name, device):
    import torch
    from lightning_indexer_top_gb300 import workloads
    from lightning_indexer_top_gb300.pipeline import SparseAttentionStep
    wa, wk, sk = WORKLOADS[name]
    wl = workloads.make(*wa, device=device, **wk)
    out_dtype = torch.float32 if wl.q_attn.dtype == torch.float32 else torch.bfloat16
    return wl, SparseAttentionStep(wl, out_dtype=out_dtype, **sk)


def parity_rows(wl):
    """Query rows the bench's parity sample checks: every row of a decode batch; for a prefill,
    every 256th row plus the first rows past the budget and the last row."""
    if wl.kind != "prefill":
        return list(range(wl.B * wl.T))
    rows = set(range(0, wl.T, 256)) | {wl.top_k - 1, wl.top_k, wl.top_k + 1, wl.T - 1}
    return sorted(r for r in rows if r < wl.T)


def config_line(name, device, steps, warmup, hbm, bf16, peak_kind, with_oracle):
    import torch
    wl, step = make_step(name, device)
    stream = torch.cuda.current_stream()
    windows, ms, _ = time_step(step, stream, steps, warmup, min_ms=200.0)
    import lightning_indexer_top_gb300 as L
    status = L.idx_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"{name}: device status {status}")
    rl, dom = rooflines(wl, step, ms, hbm, bf16, peak_kind)
    units = wl.B * wl.T
    ms_step = statistics.median(windows)
    rec = {"unit": "query tokens/s" if wl.kind == "prefill" else UNIT, "value": units / (ms_step * 1e-3),
           "ms_per_step": ms_step, "ms_per_step_min": min(windows), "ms_per_step_max": max(windows),
           "windows": len(windows), "steps_per_window": steps, "ms_per_kernel": ms, "dominant": dom,
           "roofline": rl[dom], "rooflines": rl}
    if wl.kind == "prefill":
        rec["scoring_tensor_frac"] = rl["score"]["frac"]
    if with_oracle:
        dt, par = oracle_parity(wl, step, parity_rows(wl))
        rec["parity"] = par
    del step, wl
    torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration lines")
    ap.add_argument("--min-timed-ms", type=float, default=1500.0,
                    help="repeat the K-step window until this much work is timed (clock samples under load)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOADS))
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import lightning_indexer_top_gb300 as L

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    L.build() if rank == 0 else None
    if dist:
        dist.barrier()
    L.load()
    device = f"cuda:{local}"
    hbm, bf16, peak_kind = _peaks()

    wl, step = make_step(args.workload, device)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    windows, ms, (th0, th1) = time_step(step, stream, args.steps, args.warmup, args.min_timed_ms)
    if dist:
        dist.barrier()
    clocks = sampler.stop(th0, th1)
    status = L.idx_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed region")
    ms_step = max_over_ranks(statistics.median(windows), dist, torch.device("cuda", local))

    # ---- end to end through the public API with pinned host buffers.  Two
    # input/output buffer sets: while step i computes, step i+1's inputs are
    # copied in on one side stream and step i-1's result is copied out on
    # another (the double buffering of a serving loop).  Every step still
    # moves its own inputs host->device and its own result device->host
    # inside the timed region.
    from lightning_indexer_top_gb300.pipeline import SparseAttentionStep
    host_in = [wl.q_idx.cpu().pin_memory(), wl.w.cpu().pin_memory(), wl.q_attn.cpu().pin_memory()]
    wl2 = dataclasses.replace(wl, q_idx=torch.empty_like(wl.q_idx), w=torch.empty_like(wl.w),
                              q_attn=torch.empty_like(wl.q_attn))
    steps2 = [step, SparseAttentionStep(wl2, out_dtype=step.out.dtype)]
    dev_in = [[wl.q_idx, wl.w, wl.q_attn], [wl2.q_idx, wl2.w, wl2.q_attn]]
    host_out = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()   # noqa: E731
    in_ready, computed, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def e2e_run(n):
        for i in range(n):
            j = i & 1
            st = steps2[j]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(computed[j])      # step i-2 has read these inputs
                for h, d in zip(host_in, dev_in[j]):
                    d.copy_(h, non_blocking=True)
                in_ready[j].record(s_in)
            stream.wait_event(in_ready[j])
            if i >= 2:
                stream.wait_event(out_done[j])        # step i-2's result has been copied out
            st.run()
            computed[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(computed[j])
                host_out[j].copy_(st.out, non_blocking=True)
                out_done[j].record(s_out)
        for j in range(2):
            stream.wait_event(out_done[j])

    e2e_run(4)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, torch.device("cuda", local))
    del steps2, wl2

    if rank != 0:
        dist.destroy_process_group() if dist else None
        return

    B = wl.B * wl.T                       # query rows per step
    rl, dom = rooflines(wl, step, ms, hbm, bf16, peak_kind)
    roofline = dict(rl[dom])
    src = os.path.join(ROOT, "lightning_indexer_top_gb300", "csrc", "k_score_tc.cu")
    per_key = (NCU_TRAFFIC.get((_sha(src), "f16" if wl.k8 is None else "q8"))
               if (dom == "score" and wl.kind == "decode" and wl.block_size <= 1) else None)
    roofline["traffic"] = per_key * sum(wl.n_kv_host) if per_key is not None else None
    key_bytes = sum(wl.n_kv_host) * (wl.d * 2 if wl.k8 is None else wl.d + 4)
    value = job_value(ws, B, ms_step)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16/bf16 (f32 accumulate)",
        "data": "synthetic (seeded N(0,1) q/k/latent, w ~ N(0,1/64))",
        "config": {"workload": args.workload, "queries_per_gpu": B, "n_kv": max(wl.n_kv_host), "top_k": wl.top_k,
                   "indexer": "%d heads x %d, %s cache%s" % (
                       wl.H, wl.d, "int8 + f32 row scale" if wl.k8 is not None else
                       str(wl.k_idx.dtype).replace("torch.", ""), ", Hadamard" if wl.hadamard else ""),
                   "attention": ("MLA %d heads, %d/%d bf16" % (wl.q_attn.shape[1], wl.k_attn.shape[-1], wl.dv)
                                 if wl.v_attn is None else "GQA %d q / %d kv heads, %d/%d bf16" % (
                                     wl.q_attn.shape[1], wl.k_attn.shape[1], wl.k_attn.shape[-1], wl.dv)),
                   "l2": "inputs larger than L2 (key cache %.2f GB, latent %.2f GB), no flush"
                         % (wl.k_idx.numel() * 2 / 1e9, wl.k_attn.numel() * 2 / 1e9)},
        "timing": {"windows": len(windows), "steps_per_window": args.steps,
                   "ms_per_step_median": statistics.median(windows), "ms_per_step_min": min(windows),
                   "ms_per_step_max": max(windows),
                   "per_kernel": "medians over one extra window with an event between consecutive calls"},
        "key_cache_gbs": key_bytes / ((ms["score"] + ms["topk"]) * 1e-3) / 1e9,
        "key_cache_frac": key_bytes / ((ms["score"] + ms["topk"]) * 1e-3) / 1e9 / hbm,
        "ms_per_kernel": ms,
        "roofline": roofline,
        "rooflines": rl,
        "e2e": {"value": job_value(ws, B, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "double-buffered: inputs of step i+1 and the result of step i-1 copy on side streams"},
        "gpu_launches": step.launches_per_step() * args.steps * len(windows),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1:
        import oracle.cpp as C
        dt, par = oracle_parity(wl, step, parity_rows(wl))
        line["cpu_baseline"] = {"value": par["rows"] / dt, "unit": UNIT if wl.kind != "prefill" else "query tokens/s",
                                "cores": C.threads(), "kind": "oracle (C++17, OpenMP over query rows)",
                                "sample": f"{par['rows']} of the {B} query rows of one step: double-precision "
                                          "score, top-k and attention, inputs read as stored"}
        line["parity"] = par
    del step, wl
    torch.cuda.empty_cache()
    if not args.no_configs and ws == 1:
        cfgs = {}
        for name in CONFIG_LINES:
            if name == args.workload:
                continue
            cfgs[name] = config_line(name, device, args.steps, args.warmup, hbm, bf16, peak_kind,
                                     with_oracle=not args.no_cpu_baseline)
        line["configs"] = cfgs
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
