#!/usr/bin/env python3
"""Throughput of one decode step of lightning-indexer sparse attention.

Workload (one step): 64 decode queries, each over n_kv = 131072 cached tokens:
score every key with the 64-head x 128-dim indexer (F16 key cache), select
top_k = 2048 keys per query, and run MLA attention (128 heads, 576-wide bf16
latent, 512-wide value) over the selected keys.  Synthetic, seeded data.

Prints ONE JSON line (rank 0):
  value       queries/s, device-resident inputs, CUDA events over K steps
  e2e         the same metric through the public API with pinned host buffers:
              per step H2D of the step's query inputs and D2H of its output
  roofline    the dominant kernel (the indexer key-cache scan) against the
              measured HBM copy bandwidth
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

`--impl reference` times the CPU oracle instead (the reference arm).
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

# name -> (workloads.make arguments); the first is the headline the bench line reports.
# The others serve profiling captures on smaller cases and the per-config timings.
WORKLOADS = {
    "decode_mla_64x131072": (("headline",), {}),
    "decode_mla_8x131072": (("headline",), {"batch_override": 8}),
    "decode_mla_8x8192": ((2,), {}),
    "decode_mla_64x8192": (("headline",), {"n_kv_override": 8192}),
    "long_decode_mla_ragged": ((5,), {}),
    "decode_mla_64x131072_q8": (("headline",), {"quantized_keys": True}),
    "decode_mla_64x131072_paged": (("headline",), {"page_size": 64}),
    "prefill_mla_16384": ((3,), {}),
    "prefill_mla_4096": ((3,), {"n_tokens_override": 4096}),
}

# DRAM bytes of the scorer per key from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch over 8 rows x 131072 keys, scaled to a launch by
# the keys it scans), keyed by the SHA-256 of the kernel source it was taken on.  A
# source change makes the figure stale and the bench reports traffic = null.
NCU_TRAFFIC = {
    "a80fbcefa16f962c546b227806acdd9bc43f957be944ddf1aeb7b3c9f8e1917b": (268670208 + 5784576) / (8 * 131072),
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
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


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


def _threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_oracle_queries(wl, rows):
    """Run the CPU oracle (score -> select -> attend) for the given decode rows; return (seconds, selections)."""
    import numpy as np
    import torch
    import oracle as O
    import lightning_indexer_top_gb300 as L
    sels = {}
    inputs = []
    for r in rows:
        row0, n = wl.row0(r), wl.n_kv_host[r]
        rows = wl.rows_of(r, n).to(wl.k_idx.device)   # position order (through the page table if paged)
        if wl.k8 is not None:   # the quantized cache as it represents the keys
            sc = wl.k_scale[rows] if wl.k_scale is not None else L.inline_scales(wl.k8[rows], wl.d)
            keys = O.dequantize_rows(wl.k8[rows][:, :wl.d].cpu().numpy(), sc.cpu().numpy())
        else:
            keys = wl.k_idx[rows].to("cpu", torch.float64).numpy()
        inputs.append((r, wl.q_idx[r].to("cpu", torch.float64).numpy(), wl.w[r].to("cpu", torch.float64).numpy(),
                       keys,
                       wl.q_attn[r].to("cpu", torch.float64).numpy(),
                       wl.k_attn[rows].to("cpu", torch.float64).numpy(), n))
    t0 = time.perf_counter()
    for r, q, w, k, qa, lat, n in inputs:
        s, sel, out = O.decode_pipeline_mla(q, w, k, n, wl.top_k, qa, lat, wl.scale, wl.dv)
        sels[r] = (s, sel)
    return time.perf_counter() - t0, sels


def run_reference(args):
    """Reference arm: the CPU oracle, as it stands, on bounded samples of the workload."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch
    from lightning_indexer_top_gb300 import workloads
    wl = workloads.make("headline", device="cpu", batch_override=1)
    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        cpu_oracle_queries(wl, [0])
    t = 0.0
    for _ in range(args.steps):
        dt, _ = cpu_oracle_queries(wl, [0])
        t += dt
    v = args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs)",
            "config": {"workload": WORKLOAD, "sample": "1 query of the workload per step",
                       "top_k": 2048, "n_kv": 131072},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _threads(), "kind": "oracle",
                             "sample": "1 decode query (n_kv=131072) per step: score, top-k, MLA attention"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=4, help="decode queries the CPU baseline runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(WORKLOADS))
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import lightning_indexer_top_gb300 as L
    from lightning_indexer_top_gb300 import workloads
    from lightning_indexer_top_gb300.pipeline import SparseAttentionStep

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

    wa, wk = WORKLOADS[args.workload]
    wl = workloads.make(*wa, device=f"cuda:{local}", **wk)
    step = SparseAttentionStep(wl, out_dtype=torch.bfloat16)
    stream = torch.cuda.current_stream()

    # per-kernel events: (rotate) / score / select / attend of every timed step
    rotates = step.q_rot is not None

    def timed_step(ev):
        # one event between consecutive kernels (a rotate event only when there is a rotation)
        if rotates:
            ev[0].record(stream)
            step.rotate()
        ev[1].record(stream)
        step.score()
        ev[2].record(stream)
        step.select()
        ev[3].record(stream)
        step.attend()
        ev[4].record(stream)

    for _ in range(max(args.warmup, 3)):
        step.run()
    torch.cuda.synchronize()
    L.idx_device_status(reset=True)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        timed_step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    status = L.idx_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed region")

    ms_total = t_start.elapsed_time(t_end)
    ms_rotate = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) if rotates else 0.0
    ms_score = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    ms_select = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    ms_attend = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    ms_step = max_over_ranks(ms_total / args.steps, dist, torch.device("cuda", local))

    # ---- end to end through the public API with pinned host buffers.  Two
    # input/output buffer sets: while step i computes, step i+1's inputs are
    # copied in on one side stream and step i-1's result is copied out on
    # another (the double buffering of a serving loop).  Every step still
    # moves its own inputs host->device and its own result device->host
    # inside the timed region.
    host_in = [wl.q_idx.cpu().pin_memory(), wl.w.cpu().pin_memory(), wl.q_attn.cpu().pin_memory()]
    wl2 = dataclasses.replace(wl, q_idx=torch.empty_like(wl.q_idx), w=torch.empty_like(wl.w),
                              q_attn=torch.empty_like(wl.q_attn))
    steps2 = [step, SparseAttentionStep(wl2, out_dtype=torch.bfloat16)]
    dev_in = [[wl.q_idx, wl.w, wl.q_attn], [wl2.q_idx, wl2.w, wl2.q_attn]]
    host_out = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
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

    if rank != 0:
        dist.destroy_process_group() if dist else None
        return

    B = wl.B * wl.T                       # query rows per step
    hbm, bf16, peak_kind = _peaks()
    src = os.path.join(ROOT, "lightning_indexer_top_gb300", "csrc", "k_score_tc.cu")
    if wl.kind == "prefill":
        # causal scoring: sum over rows of (visible keys) x H x d multiply-adds
        n_kv_total = sum(min(t + 1, wl.n_kv_host[0]) for t in range(wl.T)) * wl.B
        key_bytes = wl.k_idx.numel() * wl.k_idx.element_size()
        flops = 2.0 * n_kv_total * wl.H * wl.d
        roofline = {"bound": "tensor", "kernel": "idx_score (prefill, tcgen05)",
                    "achieved": flops / (ms_score * 1e-3) / 1e12, "peak": bf16, "peak_kind": peak_kind,
                    "unit": "TFLOP/s", "frac": flops / (ms_score * 1e-3) / 1e12 / bf16, "traffic": None,
                    "algorithmic_flops_per_launch": flops}
    else:
        n_kv_total = sum(wl.n_kv_host)
        # bytes of one cached key: 2 per element (F16), or 1 per element + a 4-byte scale (int8 cache;
        # the inline layout's 12 bytes of row padding are not counted)
        key_bytes = n_kv_total * (wl.d * 2 if wl.k8 is None else wl.d + 4)
        # scorer's algorithmic bytes per launch: every key row read once, one f32 score written per
        # key, the queries and weights read once
        score_bytes = key_bytes + n_kv_total * 4 + B * wl.H * wl.d * 2 + B * wl.H * 4
        achieved = score_bytes / (ms_score * 1e-3) / 1e9
        per_key = NCU_TRAFFIC.get(_sha(src)) if wl.k8 is None else None
        roofline = {"bound": "hbm", "kernel": "idx_score (key-cache scan)" if wl.k8 is None else
                    "idx_score_q8 (int8 key-cache scan)", "achieved": achieved, "peak": hbm,
                    "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm,
                    "traffic": per_key * n_kv_total if per_key is not None else None,
                    "algorithmic_bytes_per_launch": score_bytes}
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
                   "attention": "MLA 128 heads, 576/512 bf16",
                   "l2": "inputs larger than L2 (key cache %.2f GB, latent %.2f GB), no flush"
                         % (wl.k_idx.numel() * 2 / 1e9, wl.k_attn.numel() * 2 / 1e9)},
        "key_cache_gbs": key_bytes / ((ms_score + ms_select) * 1e-3) / 1e9,
        "ms_per_kernel": {"hadamard": ms_rotate, "score": ms_score, "topk": ms_select, "attention": ms_attend},
        "roofline": roofline,
        "e2e": {"value": job_value(ws, B, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "double-buffered: inputs of step i+1 and the result of step i-1 copy on side streams"},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and ws == 1 and wl.kind == "decode":
        rows = list(range(min(args.cpu_sample, B)))
        dt, sels = cpu_oracle_queries(wl, rows)
        same = []
        for r in rows:
            ns = int(step.n_sel[r])
            same.append(sorted(step.idx[r, :ns].tolist()) == sels[r][1].tolist())
        line["cpu_baseline"] = {"value": len(rows) / dt, "unit": UNIT, "cores": _threads(), "kind": "oracle",
                                "sample": f"{len(rows)} of the {B} decode queries (n_kv={max(wl.n_kv_host)} max), "
                                          "float64 score, top-k and MLA attention"}
        line["parity_sample"] = {"rows": len(rows), "identical_sets": int(sum(same))}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
