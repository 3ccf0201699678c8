#!/usr/bin/env python
"""Benchmark of the GQA decode + causal prefill hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = split-KV decode of one token through the attention of all 80
Llama3-70B layers over a 32K-token cache (B=1, H_q=64, H_kv=8, d=128), each
layer with its own 128 MiB K/V cache (10 GiB in all, so no call finds its K/V
in the 126 MB L2), followed by one causal prefill of an 8K prompt (same layer
shape), one decode of the ragged batch of 16 sequences in a 128K-key cache
(8 GiB of K/V) and one chunked prefill (the last 2K tokens of a 32K prompt).
The headline `value` is the decode's HBM throughput in GB/s per
gqa_attn_decode call on the 32K layer (algorithmic bytes: every valid K and
V row read once, 2*B*H_kv*S*d*2 bytes); the prefill's TFLOP/s
(4*H_q*d*sum_i(visible keys of row i)) is reported in the `prefill` object,
the ragged batch and the chunked prefill in `ragged_decode` and
`chunked_prefill`, each with its roofline.

`--impl reference` times the fp64 CPU oracle (the correctness reference, the
only "reference implementation" this method has) on the same workload, one
KV-head group per step.  Under torchrun (N > 1) every rank runs its own
independent problem (weak scaling, no collective in the data path); rank 0
prints one JSON line.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import resource
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GQA decode HBM GB/s (% of peak); causal prefill TFLOP/s (% of BF16 peak)"
DECODE_WORKLOAD = "llama70b_decode_32k"
PREFILL_WORKLOAD = "causal_prefill_8k"
RAGGED_WORKLOAD = "ragged_decode_b16"
CHUNKED_WORKLOAD = "chunked_prefill_32k"
LAYERS = 80         # decode calls per step: one per Llama3-70B layer, each its own K/V cache
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
KERNEL_SOURCES = {
    "decode_split_kernel": "gqa_attention_decode_gb300/csrc/decode_split.cu",
    "prefill_causal_kernel": "gqa_attention_decode_gb300/csrc/prefill_causal.cu",
    "prefill_pair_kernel": "gqa_attention_decode_gb300/csrc/prefill_pair.cu",
}


def prefill_kernel_name(G):
    """The prefill kernel the library runs for group size G: CTA pairs when G is
    a multiple of 4, one CTA per unit otherwise."""
    return "prefill_pair_kernel" if G % 4 == 0 else "prefill_causal_kernel"


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--parts", default="decode,prefill,ragged,chunked",
                    help="comma list of decode,prefill,ragged,chunked (all by default)")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="decode calls per step, each on its own K/V copy")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-configs", action="store_true",
                    help="one JSON line per workload (the five configurations, multi-token "
                         "and paged decode) instead of the step line")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_hash(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def recorded_traffic(kernel):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel's
    source is unchanged since it was captured; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
        if rec.get("source_sha256") == source_hash(KERNEL_SOURCES[kernel]):
            return float(rec["bytes_per_launch"])
    except Exception:
        pass
    return None


def cpu_cores_used(fn):
    """Runs fn(); returns (result, wall seconds, effective cores = cpu time / wall)."""
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    out = fn()
    wall = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    return out, wall, max(1, round(cpu / max(wall, 1e-9)))


class ClockSampler:
    """nvidia-smi sampling (100 ms) around the timed region."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.path = tempfile.mktemp(prefix="gqa_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0, t1):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        note = "samples inside the timed region"
        if not inside:  # region shorter than the sampling period: nearest samples
            before = [r for r in rows if r[0] < t0][-1:]
            after = [r for r in rows if r[0] > t1][:1]
            inside = before + after
            note = "timed region shorter than 100 ms: nearest samples on each side"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# workload arithmetic (what counts as useful work)
# ---------------------------------------------------------------------------

def decode_bytes(w, seqlens):
    """K and V rows of every valid key, read once: 2 * H_kv * d * 2 bytes per key."""
    return 2 * w.H_kv * w.d * 2 * int(sum(int(s) for s in seqlens))


def prefill_flops(w):
    """4 * H_q * d per (query, visible key) pair: Q K^T and P V, 2 flop per MAC each."""
    pairs = sum(w.q_offset + i + 1 for i in range(w.T_q)) * w.B
    return 4.0 * w.H_q * w.d * pairs


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return None
    import numpy as np
    import gqa_synth
    import oracle

    w = gqa_synth.WORKLOADS[DECODE_WORKLOAD]
    q, k, v, seqlens = gqa_synth.workload_decode_inputs(w, "cpu")
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    n_keys = w.S_max

    def step(i, n):
        kv = i % w.H_kv
        heads = slice(kv * w.G, (kv + 1) * w.G)
        return oracle.attend_rows(qn[0, heads], kn[0, kv, :n], vn[0, kv, :n], w.scale,
                                  np.full(w.G, n))

    # size the per-step sample so the whole run stays within about three minutes
    _, t1, _ = cpu_cores_used(lambda: step(0, n_keys))
    budget = 180.0 / max(1, args.steps + args.warmup)
    if t1 > budget:
        n_keys = max(64, int(n_keys * budget / t1))
    for i in range(args.warmup):
        step(i, n_keys)

    def timed():
        for i in range(args.steps):
            step(i, n_keys)
    _, wall, cores = cpu_cores_used(timed)
    bytes_per_step = 2 * w.d * 2 * n_keys
    value = bytes_per_step * args.steps / wall / 1e9
    sample = (f"one KV-head group per step (8 query heads x {n_keys} keys x d=128 of "
              f"{DECODE_WORKLOAD}, heads rotating), fp64 numpy")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv,
                   "d": w.d, "S_kv": w.S_max},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "affinity_cores": len(os.sched_getaffinity(0))},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def cpu_baseline_decode(w, q, k, v, seqlens):
    """The oracle on the host cores over the whole decode workload, repeated
    until about 10 s of work (at most 30 s)."""
    import oracle
    qn, kn, vn = q.float().cpu().numpy(), k.float().cpu().numpy(), v.float().cpu().numpy()
    sl = seqlens.cpu().numpy()
    reps = 0

    def run():
        nonlocal reps
        t0 = time.perf_counter()
        while True:
            oracle.decode(qn, kn, vn, sl, w.scale)
            reps += 1
            el = time.perf_counter() - t0
            if el >= 10.0 or el * (reps + 1) / reps > 30.0:
                break
    _, wall, cores = cpu_cores_used(run)
    value = decode_bytes(w, sl) * reps / wall / 1e9
    return {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"whole {DECODE_WORKLOAD} decode x{reps} in fp64 ({wall:.1f} s)",
            "affinity_cores": len(os.sched_getaffinity(0))}


def cpu_baseline_prefill(w, q, k, v):
    """The oracle on the last 256 rows (the longest ones) of one query head."""
    import numpy as np
    import oracle
    rows = min(256, w.T_q)
    r0 = w.T_q - rows
    n = w.q_offset + w.T_q
    qn = q[0, 0, r0:].float().cpu().numpy()
    kn = k[0, 0, :n].float().cpu().numpy()
    vn = v[0, 0, :n].float().cpu().numpy()
    vis = w.q_offset + np.arange(r0, w.T_q) + 1
    reps = 0

    def run():
        nonlocal reps
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            oracle.attend_rows(qn, kn, vn, w.scale, vis)
            reps += 1
    _, wall, cores = cpu_cores_used(run)
    flops = 4.0 * w.d * float(vis.sum()) * reps
    return {"value": flops / wall / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"last {rows} rows of query head 0 of {PREFILL_WORKLOAD} x{reps} in fp64",
            "affinity_cores": len(os.sched_getaffinity(0))}


def run_ours(args, rank, world, device):
    import torch
    import gqa_synth
    import gqa_attention_decode_gb300 as gqa
    from gqa_attention_decode_gb300 import build as gbuild

    if rank == 0 or world == 1:
        gbuild.build()
    if world > 1:
        torch.distributed.barrier()
    gqa.load_library()

    parts = set(args.parts.split(","))
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count

    # ---- decode inputs (resident in HBM before the timed region) ----
    wd = gqa_synth.WORKLOADS[DECODE_WORKLOAD]
    q, k, v, seqlens_cpu = gqa_synth.workload_decode_inputs(wd, device)
    seqlens = seqlens_cpu.to(device)
    # one K/V cache per decoded layer, so consecutive calls never find their K/V
    # in L2
    layers = max(1, args.layers)
    kv_copies = [(k, v)] + [(k.clone(), v.clone()) for _ in range(layers - 1)]
    splits, chunk = gqa.gqa_attn_decode_plan(wd.B, wd.H_kv, wd.S_max, sms, wd.num_splits)
    ws = torch.empty(gqa.gqa_attn_decode_workspace_size(wd.B, wd.H_q, wd.H_kv, wd.S_max, wd.d,
                                                        sms, wd.num_splits),
                     dtype=torch.uint8, device=device)
    o = torch.empty((wd.B, wd.H_q, wd.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((wd.B, wd.H_q), dtype=torch.float32, device=device)
    bytes_decode = decode_bytes(wd, seqlens_cpu.tolist())

    # ---- prefill inputs ----
    wp = gqa_synth.WORKLOADS[PREFILL_WORKLOAD]
    if "prefill" in parts:
        pq, pk, pv = gqa_synth.workload_prefill_inputs(wp, device)
        po = torch.empty_like(pq)
        plse = torch.empty((wp.B, wp.H_q, wp.T_q), dtype=torch.float32, device=device)
        pws = torch.empty(gqa.gqa_attn_prefill_causal_workspace_size(
            wp.B, wp.H_q, wp.H_kv, wp.T_q, wp.S_kv, wp.d, wp.q_offset,
            torch.cuda.get_device_properties(device).multi_processor_count),
            dtype=torch.uint8, device=device)
    flops_prefill = prefill_flops(wp)

    # ---- the largest workloads: ragged batch of 16, chunked 32K prefill ----
    wr = gqa_synth.WORKLOADS[RAGGED_WORKLOAD]
    if "ragged" in parts:
        rq, rk, rv, rsl_cpu = gqa_synth.workload_decode_inputs(wr, device)
        rsl = rsl_cpu.to(device)
        rws = torch.empty(gqa.gqa_attn_decode_workspace_size(wr.B, wr.H_q, wr.H_kv, wr.S_max,
                                                             wr.d, sms, wr.num_splits),
                          dtype=torch.uint8, device=device)
        ro = torch.empty((wr.B, wr.H_q, wr.d), dtype=torch.bfloat16, device=device)
        rlse = torch.empty((wr.B, wr.H_q), dtype=torch.float32, device=device)
        bytes_ragged = decode_bytes(wr, rsl_cpu.tolist())
    wc = gqa_synth.WORKLOADS[CHUNKED_WORKLOAD]
    if "chunked" in parts:
        cq, ck, cv = gqa_synth.workload_prefill_inputs(wc, device)
        co = torch.empty_like(cq)
        clse = torch.empty((wc.B, wc.H_q, wc.T_q), dtype=torch.float32, device=device)
        cws = torch.empty(gqa.gqa_attn_prefill_causal_workspace_size(
            wc.B, wc.H_q, wc.H_kv, wc.T_q, wc.S_kv, wc.d, wc.q_offset, sms),
            dtype=torch.uint8, device=device)
    flops_chunked = prefill_flops(wc)

    # kernels one gqa_attn_decode call launches: 1 (cluster-merged single kernel)
    # or 2 (split + merge); with 2, a split-only graph times the dominant kernel
    call_kernels = gqa.gqa_attn_decode_kernel_count(wd.B, wd.H_q, wd.H_kv, wd.S_max, wd.d,
                                                    wd.num_splits, device)
    launches_per_step = 0
    if "decode" in parts:
        launches_per_step += layers * call_kernels + (layers if call_kernels == 2 else 0)
    if "prefill" in parts:
        launches_per_step += gqa.gqa_attn_prefill_causal_kernel_count(
            wp.B, wp.H_q, wp.H_kv, wp.T_q, wp.S_kv, wp.d, wp.q_offset, pws.numel(), device)
    if "ragged" in parts:
        launches_per_step += gqa.gqa_attn_decode_kernel_count(wr.B, wr.H_q, wr.H_kv, wr.S_max,
                                                              wr.d, wr.num_splits, device)
    if "chunked" in parts:
        launches_per_step += gqa.gqa_attn_prefill_causal_kernel_count(
            wc.B, wc.H_q, wc.H_kv, wc.T_q, wc.S_kv, wc.d, wc.q_offset, cws.numel(), device)

    # The calls of a step are captured once into CUDA graphs; the timed loop
    # replays the graphs with timing events between them, so host overhead
    # never leaves the GPU idle inside a measured interval.
    def call_decode_layers():              # the public entry point, LAYERS layers
        for kc, vc in kv_copies:
            gqa.gqa_attn_decode(q, kc, vc, seqlens, wd.scale, wd.num_splits, o, lse, ws)

    def call_split_layers():               # the dominant kernel alone
        for kc, vc in kv_copies:
            gqa.gqa_attn_decode_split(q, kc, vc, seqlens, wd.scale, wd.num_splits, ws)

    def call_prefill():
        gqa.gqa_attn_prefill_causal(pq, pk, pv, wp.scale, wp.q_offset, po, plse, pws)

    def call_ragged():
        gqa.gqa_attn_decode(rq, rk, rv, rsl, wr.scale, wr.num_splits, ro, rlse, rws)

    def call_chunked():
        gqa.gqa_attn_prefill_causal(cq, ck, cv, wc.scale, wc.q_offset, co, clse, cws)

    calls = {}
    if "decode" in parts:
        calls["decode"] = call_decode_layers
        if call_kernels == 2:
            calls["split"] = call_split_layers
    if "prefill" in parts:
        calls["prefill"] = call_prefill
    if "ragged" in parts:
        calls["ragged"] = call_ragged
    if "chunked" in parts:
        calls["chunked"] = call_chunked
    for _ in range(max(args.warmup, 3)):          # eager warm-up (also per-device set-up)
        for fn in calls.values():
            fn()
    torch.cuda.synchronize(device)
    graphs = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs[name] = g
    for _ in range(2):                            # warm the graphs
        for g in graphs.values():
            g.replay()
    torch.cuda.synchronize(device)
    if gqa.gqa_attn_device_status(stream, device) != 0:
        raise RuntimeError("a bounded device wait ran out during warm-up")

    def step(ev):
        if "decode" in parts:
            ev[0].record(stream)
            graphs["decode"].replay()
            ev[1].record(stream)
            if "split" in graphs:
                ev[2].record(stream)
                graphs["split"].replay()
                ev[3].record(stream)
        if "prefill" in parts:
            ev[4].record(stream)
            graphs["prefill"].replay()
            ev[5].record(stream)
        if "ragged" in parts:
            ev[6].record(stream)
            graphs["ragged"].replay()
            ev[7].record(stream)
        if "chunked" in parts:
            ev[8].record(stream)
            graphs["chunked"].replay()
            ev[9].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(10)]
    gpu_id = f"GPU-{torch.cuda.get_device_properties(device).uuid}"
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    events = [mk() for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t_begin = time.time()
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")   # lets a profiler select the timed launches
    region0.record(stream)
    for i in range(args.steps):
        step(events[i])
    region1.record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    t_end = time.time()
    sampler.stop()
    clocks = sampler.summary(t_begin, t_end)
    if gqa.gqa_attn_device_status(stream, device) != 0:
        raise RuntimeError("a bounded device wait ran out in the timed region")

    region_ms = region0.elapsed_time(region1)
    decode_ms = split_ms = prefill_ms = 0.0
    if "decode" in parts:
        decode_ms = sum(e[0].elapsed_time(e[1]) for e in events) / layers
        split_ms = (sum(e[2].elapsed_time(e[3]) for e in events) / layers
                    if "split" in graphs else decode_ms)
    if "prefill" in parts:
        prefill_ms = sum(e[4].elapsed_time(e[5]) for e in events)
    ragged_ms = chunked_ms = 0.0
    if "ragged" in parts:
        ragged_ms = sum(e[6].elapsed_time(e[7]) for e in events)
    if "chunked" in parts:
        chunked_ms = sum(e[8].elapsed_time(e[9]) for e in events)
    # max over ranks of every time
    times = torch.tensor([region_ms, decode_ms, split_ms, prefill_ms, ragged_ms, chunked_ms],
                         dtype=torch.float64)
    if world > 1:
        t = times.to(device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        times = t.cpu()
    region_ms, decode_ms, split_ms, prefill_ms, ragged_ms, chunked_ms = times.tolist()
    K = args.steps
    result = {
        "metric": METRIC, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": region_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "B": wd.B, "H_q": wd.H_q, "H_kv": wd.H_kv,
                   "d": wd.d, "S_kv": wd.S_max, "num_splits": splits, "chunk_keys": chunk,
                   "prefill_workload": PREFILL_WORKLOAD if "prefill" in parts else None,
                   "ragged_workload": RAGGED_WORKLOAD if "ragged" in parts else None,
                   "chunked_workload": CHUNKED_WORKLOAD if "chunked" in parts else None,
                   "step": "+".join(p for p in ("decode", "prefill", "ragged", "chunked")
                                    if p in parts),
                   "layers_per_step": layers,
                   "l2": (f"each of the {layers} decode calls of a step reads its own 128 MiB "
                          f"K/V copy ({layers * 128} MiB rotating set)"),
                   "parallelism": f"{world} independent replicas (weak scaling)",
                   "launch": "each ABI call replayed as a captured CUDA graph"},
        "gpu_launches": launches_per_step * K,
    }
    if "decode" in parts:
        call_ms = decode_ms / K                   # one whole gqa_attn_decode call
        value = world * bytes_decode / (call_ms * 1e-3) / 1e9
        achieved = bytes_decode / (split_ms / K * 1e-3) / 1e9
        result["value"] = value
        kernel = ("decode_split_kernel (single launch, cluster merge)" if call_kernels == 1
                  else "decode_split_kernel")
        result["decode"] = {"call_us": call_ms * 1e3, "kernels_per_call": call_kernels,
                            "split_us": split_ms / K * 1e3,
                            "merge_and_gap_us": (decode_ms - split_ms) / K * 1e3,
                            "bytes_per_call": bytes_decode,
                            "frac_of_hbm_peak": value / world / peaks["hbm_gbs"],
                            "frac_of_8tbs_nominal": value / world / 8000.0}
        result["roofline"] = {"bound": "hbm", "kernel": kernel,
                              "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": achieved / peaks["hbm_gbs"],
                              "traffic": recorded_traffic("decode_split_kernel"),
                              "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    if "prefill" in parts:
        pms = prefill_ms / K
        tflops = flops_prefill / (pms * 1e-3) / 1e12
        result["prefill"] = {
            "workload": PREFILL_WORKLOAD, "value": world * tflops, "unit": "TFLOP/s",
            "us_per_call": pms * 1e3, "flops_per_call": flops_prefill,
            "roofline": {"bound": "tensor", "kernel": prefill_kernel_name(wp.G),
                         "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tflops / peaks["bf16_tflops"],
                         "frac_of_sustained": tflops / peaks["bf16_tflops_sustained"],
                         "traffic": recorded_traffic(prefill_kernel_name(wp.G)),
                         "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)"}}
        if "decode" not in parts:
            result["value"] = world * tflops
            result["unit"] = "TFLOP/s"
    if "ragged" in parts:
        rus = ragged_ms / K * 1e3
        gbs = bytes_ragged / (rus * 1e-6) / 1e9
        rk_count = gqa.gqa_attn_decode_kernel_count(wr.B, wr.H_q, wr.H_kv, wr.S_max, wr.d,
                                                    wr.num_splits, device)
        rsplits, rchunk = gqa.gqa_attn_decode_plan(wr.B, wr.H_kv, wr.S_max, sms, wr.num_splits)
        result["ragged_decode"] = {
            "workload": RAGGED_WORKLOAD, "value": world * gbs, "unit": "GB/s",
            "us_per_call": rus, "bytes_per_call": bytes_ragged, "kernels_per_call": rk_count,
            "seqlens_sum": int(rsl_cpu.sum()), "num_splits": rsplits, "chunk_keys": rchunk,
            "l2": f"{2 * rk.numel() * 2 >> 30} GiB padded K/V cache, larger than L2",
            "roofline": {"bound": "hbm", "kernel": "decode_split_kernel + decode_merge_kernel "
                         "(whole call)", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "frac_of_8tbs_nominal": gbs / 8000.0, "traffic": None,
                         "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}}
    if "chunked" in parts:
        cus = chunked_ms / K * 1e3
        ctf = flops_chunked / (cus * 1e-6) / 1e12
        result["chunked_prefill"] = {
            "workload": CHUNKED_WORKLOAD, "value": world * ctf, "unit": "TFLOP/s",
            "us_per_call": cus, "flops_per_call": flops_chunked,
            "kernels_per_call": gqa.gqa_attn_prefill_causal_kernel_count(
                wc.B, wc.H_q, wc.H_kv, wc.T_q, wc.S_kv, wc.d, wc.q_offset, cws.numel(), device),
            "roofline": {"bound": "tensor", "kernel": prefill_kernel_name(wc.G) +
                         " (+ piece merge)", "achieved": ctf, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": ctf / peaks["bf16_tflops"],
                         "frac_of_sustained": ctf / peaks["bf16_tflops_sustained"],
                         "traffic": None,
                         "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)"}}
    result["clocks"] = clocks

    # ---- end to end through the host-buffer entry points ----
    if not args.no_e2e:
        result["e2e"] = e2e_decode(args, gqa, wd, q, k, v, seqlens_cpu, sms, device, stream, world)
        if "prefill" in parts:
            result["prefill"]["e2e"] = e2e_prefill(gqa, wp, pq, pk, pv, device, stream, world,
                                                   flops_prefill)
    # ---- CPU baseline (rank 0, one GPU only) ----
    if world == 1 and not args.no_cpu_baseline:
        if "decode" in parts:
            result["cpu_baseline"] = cpu_baseline_decode(wd, q, k, v, seqlens_cpu)
        if "prefill" in parts:
            result["prefill"]["cpu_baseline"] = cpu_baseline_prefill(wp, pq, pk, pv)
            if "decode" not in parts:
                result["cpu_baseline"] = result["prefill"]["cpu_baseline"]
    return result


def e2e_decode(args, gqa, wd, q, k, v, seqlens_cpu, sms, device, stream, world):
    import torch
    qh, kh, vh = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    sh = seqlens_cpu.pin_memory()
    oh = torch.empty((wd.B, wd.H_q, wd.d), dtype=torch.bfloat16).pin_memory()
    lh = torch.empty((wd.B, wd.H_q), dtype=torch.float32).pin_memory()
    arena = torch.empty(gqa.gqa_attn_decode_from_host_arena_size(
        wd.B, wd.H_q, wd.H_kv, wd.S_max, wd.d, sms, wd.num_splits), dtype=torch.uint8,
        device=device)
    steps = max(3, min(args.steps, 50))
    for _ in range(3):
        gqa.gqa_attn_decode_from_host(qh, kh, vh, sh, wd.scale, wd.num_splits, oh, lh, arena, stream)
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        gqa.gqa_attn_decode_from_host(qh, kh, vh, sh, wd.scale, wd.num_splits, oh, lh, arena, stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    wall = _max_over_ranks(wall, world, device)
    nbytes = decode_bytes(wd, seqlens_cpu.tolist())
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2 + sh.numel() * 4
    d2h = oh.numel() * 2 + lh.numel() * 4
    return {"value": world * nbytes * steps / wall / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": "gqa_attn_decode_from_host (pinned host buffers)"}


def e2e_prefill(gqa, wp, pq, pk, pv, device, stream, world, flops):
    import torch
    qh, kh, vh = pq.cpu().pin_memory(), pk.cpu().pin_memory(), pv.cpu().pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((wp.B, wp.H_q, wp.T_q), dtype=torch.float32).pin_memory()
    arena = torch.empty(gqa.gqa_attn_prefill_causal_from_host_arena_size(
        wp.B, wp.H_q, wp.H_kv, wp.T_q, wp.S_kv, wp.d), dtype=torch.uint8, device=device)
    for _ in range(2):
        gqa.gqa_attn_prefill_causal_from_host(qh, kh, vh, wp.scale, wp.q_offset, oh, lh, arena,
                                              stream)
    torch.cuda.synchronize(device)
    steps = 10
    t0 = time.perf_counter()
    for _ in range(steps):
        gqa.gqa_attn_prefill_causal_from_host(qh, kh, vh, wp.scale, wp.q_offset, oh, lh, arena,
                                              stream)
    torch.cuda.synchronize(device)
    wall = _max_over_ranks(time.perf_counter() - t0, world, device)
    return {"value": world * flops * steps / wall / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": (qh.numel() + kh.numel() + vh.numel()) * 2,
            "d2h_bytes_per_step": oh.numel() * 2 + lh.numel() * 4, "steps": steps}


def _max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_all_configs(device):
    """Times every workload on its own (CUDA graphs of calls, CUDA events) and
    prints one JSON line each with its roofline fraction."""
    import torch
    import gqa_synth
    import gqa_attention_decode_gb300 as gqa
    from gqa_attention_decode_gb300 import build as gbuild
    gbuild.build()
    gqa.load_library()
    peaks, peak_src = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size

    def time_graph(fn, calls, reps):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize(device)
        if gqa.gqa_attn_device_status() != 0:
            raise RuntimeError("device status not OK")
        return e0.elapsed_time(e1) * 1e3 / (reps * calls)

    def emit(d):
        d["peak_source"] = peak_src
        print(json.dumps(d), flush=True)

    def decode_line(name, T_q=1, page_size=0, cache_keys=0):
        w = gqa_synth.WORKLOADS[name]
        q, k, v, sl = gqa_synth.workload_decode_inputs(w, device)
        if cache_keys:  # the same sequences inside a longer (over-allocated) cache
            q, k, v, sl = gqa_synth.decode_inputs(w.B, w.H_q, w.H_kv, cache_keys, w.d, w.seed,
                                                  device, sl.tolist())
        if T_q > 1:
            q = gqa_synth.bf16_normal((w.B, w.H_q, T_q, w.d), w.seed, device)
        nbytes = decode_bytes(w, sl.tolist())
        # enough distinct K/V copies that consecutive calls never find theirs in L2
        # (counted by the bytes a call reads: a cache longer than its sequences is
        # read only up to their lengths, and re-reading the same 128 MiB every call
        # would measure a different, L2-shared regime)
        copies = 1 if nbytes > 2 * l2_bytes else min(16, -(-(1 << 30) // nbytes))
        kvs = [(k, v)] + [(k.clone(), v.clone()) for _ in range(copies - 1)]
        sld = sl.to(device)
        ns = w.num_splits or 0
        if page_size:
            mp = w.S_max // page_size
            pages = []
            for kc, vc in kvs:
                kp = kc.view(w.B, w.H_kv, mp, page_size, w.d).permute(0, 2, 1, 3, 4).reshape(
                    w.B * mp, w.H_kv, page_size, w.d).contiguous()
                vp = vc.view(w.B, w.H_kv, mp, page_size, w.d).permute(0, 2, 1, 3, 4).reshape(
                    w.B * mp, w.H_kv, page_size, w.d).contiguous()
                pages.append((kp, vp))
            table = torch.arange(w.B * mp, dtype=torch.int32, device=device).view(w.B, mp)
            if T_q > 1:
                fn = lambda: [gqa.gqa_attn_decode_paged_multi(q, kp, vp, table, sld, w.scale, ns)
                              for kp, vp in pages]
            else:
                fn = lambda: [gqa.gqa_attn_decode_paged(q, kp, vp, table, sld, w.scale, ns)
                              for kp, vp in pages]
        elif T_q > 1:
            fn = lambda: [gqa.gqa_attn_decode_multi(q, kc, vc, sld, w.scale, ns) for kc, vc in kvs]
        else:
            fn = lambda: [gqa.gqa_attn_decode(q, kc, vc, sld, w.scale, ns) for kc, vc in kvs]
        us = time_graph(fn, len(kvs), 20)
        gbs = nbytes / us / 1e3
        label = (name + (f" T_q={T_q}" if T_q > 1 else "") +
                 (f" paged({page_size})" if page_size else "") +
                 (f" in a {cache_keys >> 10}K-key cache" if cache_keys else ""))
        emit({"workload": label, "us_per_call": us, "value": gbs, "unit": "GB/s",
              "bound": "hbm", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
              "bytes_per_call": nbytes, "kv_copies": len(kvs),
              "l2": ("K/V read per call larger than L2" if nbytes > 2 * l2_bytes else
                     f"{len(kvs)} K/V copies rotate ({len(kvs) * nbytes >> 20} MiB read)"
                     if len(kvs) * nbytes > 2 * l2_bytes else
                     "L2 resident (latency-bound)")})

    def prefill_line(name, page_size=0):
        w = gqa_synth.WORKLOADS[name]
        q, k, v = gqa_synth.workload_prefill_inputs(w, device)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H_q, w.T_q), dtype=torch.float32, device=device)
        nb = gqa.gqa_attn_prefill_causal_workspace_size(w.B, w.H_q, w.H_kv, w.T_q, w.S_kv, w.d,
                                                        w.q_offset, sms)
        ws = torch.empty(nb, dtype=torch.uint8, device=device)
        kernels = gqa.gqa_attn_prefill_causal_kernel_count(w.B, w.H_q, w.H_kv, w.T_q, w.S_kv,
                                                           w.d, w.q_offset, nb, device)
        kernel = prefill_kernel_name(w.G)
        if page_size:   # the same K/V in a pool of pages (in order), read through a block table
            mp = -(-w.S_kv // page_size)
            kp = torch.zeros((w.B * mp, w.H_kv, page_size, w.d), dtype=k.dtype, device=device)
            vp = torch.zeros_like(kp)
            for b in range(w.B):
                for i in range(mp):
                    n = min(page_size, w.S_kv - i * page_size)
                    kp[b * mp + i, :, :n] = k[b, :, i * page_size:i * page_size + n]
                    vp[b * mp + i, :, :n] = v[b, :, i * page_size:i * page_size + n]
            table = torch.arange(w.B * mp, dtype=torch.int32, device=device).view(w.B, mp)
            fn = lambda: gqa.gqa_attn_prefill_causal_paged(q, kp, vp, table, w.S_kv, w.scale,
                                                           w.q_offset, o, lse, ws)
            name = f"{name} paged({page_size})"
            # CTA pairs read pages only when every key tile is whole
            kernel = kernel if w.S_kv % 128 == 0 else "prefill_causal_kernel"
        else:
            fn = lambda: gqa.gqa_attn_prefill_causal(q, k, v, w.scale, w.q_offset, o, lse, ws)
        us = time_graph(fn, 1, 10)
        tf = prefill_flops(w) / us / 1e6
        emit({"workload": name, "us_per_call": us, "value": tf, "unit": "TFLOP/s",
              "bound": "tensor", "kernel": kernel, "kernels_per_call": kernels,
              "peak": peaks["bf16_tflops"], "frac": tf / peaks["bf16_tflops"],
              "frac_of_sustained": tf / peaks["bf16_tflops_sustained"],
              "flops_per_call": prefill_flops(w)})

    decode_line("tiny_decode")
    decode_line("llama70b_decode_32k")
    decode_line("ragged_decode_b16")
    prefill_line("causal_prefill_8k")
    prefill_line("chunked_prefill_32k")
    decode_line("llama70b_decode_32k", T_q=4)
    decode_line("llama70b_decode_32k", T_q=16)
    decode_line("llama70b_decode_32k", page_size=256)
    decode_line("llama70b_decode_32k", T_q=16, page_size=256)
    prefill_line("chunked_prefill_32k", page_size=256)
    decode_line("llama70b_decode_32k", cache_keys=131072)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if args.all_configs:
        if rank == 0:
            run_all_configs(device)
        return
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        res = run_ours(args, rank, world, device)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
