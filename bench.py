#!/usr/bin/env python
"""Benchmark of the paged KV-cache attention hot path on GB300.

One step = one pass of the hot path over one batch of the decode workload
(64 sequences, Qwen3-0.6B attention shape 16/8/128, context_lens uniform in
[512, 4096], block_size 256, blocks shuffled over a 2048-block pool):
kv_store of the step's 64 new K/V rows and the paged decode (split kernel +
log-sum-exp merge), in one call (attn_decode_paged_append, the store fused
into the decode launch).  The step is replayed from a CUDA graph (graph-safe
decode, as the serving engine runs it) over 4 independent input sets in
rotation, so no step finds its inputs in L2 (8.6 GB footprint vs 126 MB L2).
The same step as two calls (kv_store, then attn_decode_paged) is reported
beside it under "unfused".

value = algorithmic bytes of the step (K/V of every context token read once,
q, out, new rows stored, block-table entries, context_lens) / step time, in
GB/s.  The same line carries the prefill half of the metric (varlen prefill
with prefix cache, 8 prompts, Qwen3-8B heads): causal FLOPs / time, with the
prefill steps launched eagerly (the pages' engine graph-replays decode only),
and further lines: a mixed chunked-prefill + decode step, bucketed graph
decode, copy-on-write block copies, the 150 GB decode B512 sweep, the
28-layer engine-trace replay and the host scheduler step loop.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the batch (the path shards by sequence with no exchange), time = max over
ranks, value = total bytes / time ("weak" scaling).  --impl reference times
the CPU oracle (fp64 C, all host cores) on the same workload and metric.
"""
from __future__ import annotations

import argparse
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

METRIC = "paged decode attention HBM GB/s (% of peak); prefill attention TFLOP/s (% peak)"
N_SETS = 4

# DRAM bytes per launch from ncu (dram__bytes_read.sum + dram__bytes_write.sum)
# for the dominant kernels, with the sha256 of the kernel source they were
# measured on; a figure whose source has changed since is reported as null.
TRAFFIC = {
    # decode B64 workload (one input set), one ncu --set full capture of the split kernel
    "decode": {"file": "paged_kv_cache_125_gb300/csrc/decode.cu",
               "sha256": "07f434c766015d559ae0affb2f61e9797e9003a251cbb795c3e28b4c04ea3955",
               "bytes": 569347584 + 3980544},
    # decode B512 mix: one capture of the tensor-core split kernel on 128 of the sequences
    # (1789.71 MB for 1778.58 MB algorithmic), scaled to the 512-sequence launch by its algorithmic
    # bytes (7062.70 MB)
    "decode_b512": {"file": "paged_kv_cache_125_gb300/csrc/decode.cu",
                    "sha256": "07f434c766015d559ae0affb2f61e9797e9003a251cbb795c3e28b4c04ea3955",
                    "bytes": 7106903694},
    # prefill workload (8 prompts, 32/8/128), one ncu --set full capture of the prefill kernel of
    # attn_prefill_varlen_append
    "prefill": {"file": "paged_kv_cache_125_gb300/csrc/prefill.cu",
                "sha256": "87f871db8ebb10db8884dfb6f61e8fbd782b1ab78e6e3c724783916fafdec3e9",
                "bytes": 111977728 + 33583360},
    # decode 64/8/128 on the decode B64 batch, one ncu --set full capture of the split kernel
    "decode_group8": {"file": "paged_kv_cache_125_gb300/csrc/decode.cu",
                      "sha256": "07f434c766015d559ae0affb2f61e9797e9003a251cbb795c3e28b4c04ea3955",
                      "bytes": 576161024 + 5634304},
    # the mixed step (one attn_mixed_step call): dram bytes of its four kernels (narrow store,
    # prefill, tensor-core decode, merge) from one ncu --metrics capture, summed
    "mixed": {"file": ["paged_kv_cache_125_gb300/csrc/api.cu", "paged_kv_cache_125_gb300/csrc/prefill.cu",
                       "paged_kv_cache_125_gb300/csrc/decode.cu", "paged_kv_cache_125_gb300/csrc/kv_store.cu"],
              "sha256": ["67530d107bbd4d9366bf0e741036ab01295e5defadb3a6051ddf6a63b3bea151",
                         "87f871db8ebb10db8884dfb6f61e8fbd782b1ab78e6e3c724783916fafdec3e9",
                         "07f434c766015d559ae0affb2f61e9797e9003a251cbb795c3e28b4c04ea3955",
                         "3de4572fdae061866219311055c3a52252d20b51b0cd3367ae6c4c0e416b6024"],
              "bytes": 1280745472},
    # kv_copy_blocks on the 64-pair, 56-plane call, one ncu --metrics capture
    "copy_blocks": {"file": "paged_kv_cache_125_gb300/csrc/copy_blocks.cu",
                    "sha256": "4257c5bb2346e1bde3299c7f093b29e7939976617646de065c32796c7035dea2",
                    "bytes": 1859943680 + 1831985920},
    # the prefill workload's suffix store (8150 rows), one ncu capture of kv_store_kernel
    # (SpeedOfLight + MemoryWorkloadAnalysis: dram__bytes.sum.per_second x gpu__time_duration.sum)
    "kv_store": {"file": "paged_kv_cache_125_gb300/csrc/kv_store.cu",
                 "sha256": "3de4572fdae061866219311055c3a52252d20b51b0cd3367ae6c4c0e416b6024",
                 "bytes": 34464000},
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--prefill-steps", type=int, default=None)
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-copy-blocks", action="store_true")
    p.add_argument("--no-large", action="store_true", help="skip the 150 GB decode B512 line")
    p.add_argument("--no-trace", action="store_true", help="skip the engine-trace replay line")
    p.add_argument("--only", choices=["decode", "prefill", "decode_b512", "decode_group8", "mixed",
                                      "copy_blocks", "decode_bucketed", "engine_trace"], default=None,
                   help="run one part only (profiling); the JSON line then carries that part")
    p.add_argument("--b512-batch", type=int, default=512,
                   help="sequences of the decode B512 line (a smaller batch profiles the same kernel)")
    p.add_argument("--b512-blocks", type=int, default=None,
                   help="pool blocks of the decode B512 line (default: the 150 GB pool)")
    p.add_argument("--sets", type=int, default=N_SETS, help="input sets in rotation")
    return p.parse_args()


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def traffic_for(name):
    """The entry's bytes while every source it was captured from is unchanged, else None."""
    t = TRAFFIC[name]
    if t["bytes"] is None or t["sha256"] is None:
        return None
    files = t["file"] if isinstance(t["file"], list) else [t["file"]]
    shas = t["sha256"] if isinstance(t["sha256"], list) else [t["sha256"]]
    for f, sha in zip(files, shas):
        if hashlib.sha256(open(os.path.join(ROOT, f), "rb").read()).hexdigest() != sha:
            return None
    return t["bytes"]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, windows=()):
        """Summary of the samples taken inside the given (t0, t1) windows."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if windows and not any(t0 <= ts <= t1 for t0, t1 in windows):
                continue
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads

def decode_bytes(w):
    """Algorithmic bytes of one step: (store) read k, v rows + write them into
    the cache; (decode) K and V of every context token once, q, out, the used
    block-table entries and context_lens."""
    a = w.steps[0].attn.meta
    b = a.context_lens.numel()
    row = w.num_kv_heads * w.head_dim * 2
    ctx = a.context_lens.long()
    store = 4 * b * row
    kv = int(ctx.sum()) * row * 2
    qo = 2 * b * w.num_heads * w.head_dim * 2
    tables = int(((ctx + w.block_size - 1) // w.block_size).sum()) * 4 + b * 4
    return store, kv + qo + tables


def prefill_flops(w):
    m = w.steps[0].attn.meta
    q = (m.cu_seqlens_q[1:] - m.cu_seqlens_q[:-1]).long()
    k = (m.cu_seqlens_k[1:] - m.cu_seqlens_k[:-1]).long()
    c = k - q
    visible = int((q * c + q * (q + 1) // 2).sum())
    return 4 * w.head_dim * w.num_heads * visible


class DeviceSet:
    """One resident copy of a workload's step inputs and cache on the device."""

    def __init__(self, w, device):
        import torch
        kc, vc = w.new_cache(device, poison=True)
        w.place_history(kc, vc)
        for st in w.setup:
            self._store(st, kc, vc, device)
        step = w.steps[0]
        s, a = step.store, step.attn
        self.k, self.v = s.k.to(device), s.v.to(device)
        self.slots = s.slot_mapping.to(device)
        self.q = a.q.to(device)
        self.kc, self.vc = kc, vc
        m = a.meta
        if step.is_prefill:
            self.cu_q, self.cu_k = m.cu_seqlens_q.to(device), m.cu_seqlens_k.to(device)
            self.max_q, self.max_k = m.max_seqlen_q, m.max_seqlen_k
            self.bt = None if m.block_tables is None else m.block_tables.to(device)
            self.out = torch.empty_like(self.q)
        else:
            self.bt, self.ctx = m.block_tables.to(device), m.context_lens.to(device)
            self.max_ctx = m.max_context_len
            self.out = torch.empty_like(self.q)

    @staticmethod
    def _store(st, kc, vc, device):
        import paged_kv_cache_125_gb300 as kvp
        kvp.kv_store(st.k.to(device), st.v.to(device), st.slot_mapping.to(device), kc, vc)


def store_call(kvp, s):
    kvp.kv_store(s.k, s.v, s.slots, s.kc, s.vc)


def decode_call(kvp, s, w, ws):
    kvp.attn_decode_paged(s.q, s.kc, s.vc, s.bt, s.ctx, s.max_ctx, softmax_scale=w.scale,
                          workspace=ws, out=s.out)


def append_call(kvp, s, w, ws):
    """The decode step in one call: kv_store of the new rows fused into the decode."""
    kvp.attn_decode_paged_append(s.q, s.k, s.v, s.slots, s.kc, s.vc, s.bt, s.ctx, s.max_ctx,
                                 softmax_scale=w.scale, workspace=ws, out=s.out)


def prefill_append_call(kvp, s, w):
    """The prefill step in one call: the store of the new rows fused into the prefill."""
    kvp.attn_prefill_varlen_append(s.q, s.k, s.v, s.slots, s.cu_q, s.cu_k, s.max_q, s.max_k, s.kc, s.vc,
                                   block_tables=s.bt, softmax_scale=w.scale, out=s.out)


def no_call(s):
    pass


def prefill_call(kvp, s, w):
    kvp.attn_prefill_varlen(s.q, s.cu_q, s.cu_k, s.max_q, s.max_k, k=s.k, v=s.v, k_cache=s.kc,
                            v_cache=s.vc, block_tables=s.bt, num_kv_heads=w.num_kv_heads,
                            softmax_scale=w.scale, out=s.out)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Largest value of x over all ranks (per-step time: the slowest rank
    defines the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_units, ms_per_rank, world, device="cuda"):
    """Whole-job throughput of `world` replicas that each process step_units
    per step: total units / max-over-ranks step time (units per second)."""
    ms = max_over_ranks(ms_per_rank, world, device)
    return step_units * world / (ms * 1e-3), ms


def capture(fn, sets, stream):
    """One CUDA graph per input set for the callable fn(set)."""
    import torch
    graphs = []
    for s in sets:
        fn(s)  # first use outside capture (library set-up)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn(s)
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


def timed_loop(store_graphs, attn_graphs, steps, warmup, world):
    """One step = store graph + attention graph of input set i % n.  K steps
    are timed between barrier + synchronize pairs; an event pair around every
    attention graph (on the launching stream, outside the graphs) gives the
    attention call's duration inside the timed region.
    Returns (ms per step, mean ms of the attention call, wall window)."""
    import torch
    n = len(store_graphs)
    for i in range(warmup):
        store_graphs[i % n].replay()
        attn_graphs[i % n].replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    start.record()
    for i in range(steps):
        store_graphs[i % n].replay()
        evs[i][0].record()
        attn_graphs[i % n].replay()
        evs[i][1].record()
    stop.record()
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    barrier(world)
    ms_step = start.elapsed_time(stop) / steps
    durs = [a.elapsed_time(b) for a, b in evs]
    return ms_step, statistics.mean(durs), (w0, w1)


def timed_loop_single(graphs, steps, warmup, world):
    """One step = one graph replay of input set i % n (the fused store +
    decode call); an event pair around every replay gives the call's duration.
    Returns (ms per step, mean ms of the call, wall window)."""
    import torch
    n = len(graphs)
    for i in range(warmup):
        graphs[i % n].replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    start.record()
    for i in range(steps):
        evs[i][0].record()
        graphs[i % n].replay()
        evs[i][1].record()
    stop.record()
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    barrier(world)
    ms_step = start.elapsed_time(stop) / steps
    durs = [a.elapsed_time(b) for a, b in evs]
    return ms_step, statistics.mean(durs), (w0, w1)


def timed_loop_eager(store_fn, attn_fn, sets, steps, warmup, world, call_events=True):
    """As timed_loop, with the two calls launched directly (no graph): the
    pages' engine runs prefill steps eagerly and graph-replays only decode.
    Without call_events nothing is recorded between the steps (an event
    record between two launches stops the second from starting early as a
    programmatic dependent); the mean call time is then None."""
    import torch
    n = len(sets)
    for i in range(warmup):
        store_fn(sets[i % n])
        attn_fn(sets[i % n])
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    start.record()
    for i in range(steps):
        if call_events:
            evs[i][0].record()
        store_fn(sets[i % n])
        if call_events:
            evs[i][1].record()
        attn_fn(sets[i % n])
        if call_events:
            evs[i][2].record()
    stop.record()
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    barrier(world)
    ms_step = start.elapsed_time(stop) / steps
    if not call_events:
        return ms_step, None, (w0, w1)
    durs = [b.elapsed_time(c) for a, b, c in evs]
    timed_loop_eager.last_store_ms = statistics.mean(a.elapsed_time(b) for a, b, c in evs)
    return ms_step, statistics.mean(durs), (w0, w1)


# ----------------------------------------------------------------------------- CPU oracle

def oracle_decode_rate(w, min_seconds=8.0):
    """The oracle (fp64 C, all host cores) on the whole decode step (store +
    decode of all 64 sequences), repeated until min_seconds have passed."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from parity import oracle_pool
    kc, vc = oracle_pool(w)
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta
    q_cpu = a.q.cpu()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.kv_store(st.k.cpu(), st.v.cpu(), st.slot_mapping.cpu(), kc, vc)
        oracle.decode(q_cpu, kc, vc, m.block_tables, m.context_lens, w.num_heads, w.num_kv_heads,
                      w.scale)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    store, dec = decode_bytes(w)
    return (store + dec) * reps / el / 1e9, el / reps, reps, oracle.num_threads()


# ----------------------------------------------------------------------------- main arms

def bench_config(w, sets):
    """The config dict both arms print: the workload and how the timed steps
    avoid L2 reuse (input sets in rotation whose pools exceed the L2)."""
    pools_gb = w.num_blocks * w.block_size * w.num_kv_heads * w.head_dim * 2 * 2 * sets / 1e9
    return {"workload": w.description,
            "l2": f"{sets} input sets in rotation ({pools_gb:.1f} GB of pools) vs 126 MB L2"}


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores, on the same workload and
    metric: each step is the full decode step (store + decode of all 64
    sequences); --warmup untimed steps (at least 3, then up to ~20 s), then at
    most --steps steps and about 60 s of timed work."""
    if rank != 0:
        return
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from parity import oracle_pool
    from paged_kv_cache_125_gb300 import workloads as W
    w = W.config2_decode()
    kc, vc = oracle_pool(w)
    st, a = w.steps[0].store, w.steps[0].attn
    m = a.meta

    def step():
        oracle.kv_store(st.k, st.v, st.slot_mapping, kc, vc)
        oracle.decode(a.q, kc, vc, m.block_tables, m.context_lens, w.num_heads, w.num_kv_heads, w.scale)

    warm, tw = 0, time.perf_counter()
    while warm < args.warmup and (warm < 3 or time.perf_counter() - tw < 20.0):
        step()
        warm += 1
    done, t0 = 0, time.perf_counter()
    while done < args.steps and (done == 0 or time.perf_counter() - t0 < 60.0):
        step()
        done += 1
    el = time.perf_counter() - t0
    store, dec = decode_bytes(w)
    value = (store + dec) * done / el / 1e9
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": done, "warmup": warm,
            "ms_per_step": round(1000 * el / done, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, args.sets),
            "parallelism": f"{cores} host threads",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"full decode step (store + decode of all 64 sequences) x {done}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_decode(args, kvp, W, dev, stream, world, peaks):
    import torch
    w = W.config2_decode()
    store_b, dec_b = decode_bytes(w)
    step_bytes = store_b + dec_b
    sets = [DeviceSet(w, dev) for _ in range(args.sets)]
    ws = torch.empty(kvp.attn_decode_workspace_size(64, w.num_heads, w.head_dim,
                                                    w.steps[0].attn.meta.max_context_len,
                                                    w.block_size), dtype=torch.uint8, device=dev)
    app_graphs = capture(lambda s: append_call(kvp, s, w, ws), sets, stream)
    assert kvp.device_status() == 0
    ms_step, ms_call, win = timed_loop_single(app_graphs, args.steps, args.warmup, world)
    assert kvp.device_status() == 0, "device status after the timed decode loop"
    bytes_per_s, ms_step = aggregate(step_bytes, ms_step, world)
    achieved = step_bytes / (ms_call * 1e-3) / 1e9
    res = {"w": w, "window": win, "ms_step": ms_step, "value": bytes_per_s / 1e9,
           "roofline": {"kernel": "attn_decode_paged_append (store + split + merge)", "bound": "hbm",
                        "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic_for("decode"),
                        "algorithmic_bytes": step_bytes, "peak_source": peaks["source"],
                        "ms_per_launch": round(ms_call, 5)}}

    # the same step as two calls (kv_store graph, then attn_decode_paged graph)
    store_graphs = capture(lambda s: store_call(kvp, s), sets, stream)
    dec_graphs = capture(lambda s: decode_call(kvp, s, w, ws), sets, stream)
    ms_ustep, ms_decode, uwin = timed_loop(store_graphs, dec_graphs, args.steps, args.warmup, world)
    assert kvp.device_status() == 0, "device status after the unfused decode loop"
    ubps, ms_ustep = aggregate(step_bytes, ms_ustep, world)
    dec_achieved = dec_b / (ms_decode * 1e-3) / 1e9
    res["unfused"] = {"step": "kv_store graph + attn_decode_paged graph", "value": round(ubps / 1e9, 2),
                      "unit": "GB/s", "ms_per_step": round(ms_ustep, 5), "steps": args.steps,
                      "decode_call": {"kernel": "attn_decode_paged (split + merge)",
                                      "achieved": round(dec_achieved, 1), "unit": "GB/s",
                                      "frac": round(dec_achieved / peaks["hbm_gbs"], 4),
                                      "algorithmic_bytes": dec_b, "ms_per_launch": round(ms_decode, 5)}}
    res["uwindow"] = uwin
    del store_graphs, dec_graphs

    # end to end through the API with host buffers (pinned), per step: the
    # step's inputs (q, new k/v rows, slots, block tables, context lens) sit in
    # one packed pinned buffer and travel in one host->device copy into one
    # packed device buffer, whose views the captured step reads.
    import types
    s0 = sets[0]
    parts = [s0.q, s0.k, s0.v, s0.slots, s0.bt, s0.ctx]
    offs, nbytes = [], 0
    for t in parts:
        nbytes = (nbytes + 255) // 256 * 256
        offs.append(nbytes)
        nbytes += t.numel() * t.element_size()
    dev_pack = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    host_pack = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)

    def view(buf, t, o):
        return buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    dv = [view(dev_pack, t, o) for t, o in zip(parts, offs)]
    for t, o in zip(parts, offs):
        view(host_pack, t, o).copy_(t.cpu())
    es = types.SimpleNamespace(q=dv[0], k=dv[1], v=dv[2], slots=dv[3], bt=dv[4], ctx=dv[5],
                               kc=s0.kc, vc=s0.vc, max_ctx=s0.max_ctx, out=torch.empty_like(s0.out))
    dev_pack.copy_(host_pack)
    e2e_graph = capture(lambda s_: append_call(kvp, s_, w, ws), [es], stream)[0]
    host_out = torch.empty(es.out.shape, dtype=es.out.dtype, pin_memory=True)
    h2d = host_pack.numel()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        dev_pack.copy_(host_pack, non_blocking=True)
        e2e_graph.replay()
        host_out.copy_(es.out, non_blocking=True)
        stream.synchronize()

    for _ in range(5):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    e2e_bps, e2e_ms = aggregate(step_bytes, e2e_ms, world)
    res["e2e"] = {"value": round(e2e_bps / 1e9, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                  "how": "packed pinned host inputs copied in (one copy), graph replay, output copied "
                         "out, stream sync each step"}
    del app_graphs, sets, e2e_graph
    return res


def measure_prefill(args, kvp, W, dev, stream, world, peaks):
    """The prefill configuration (8 prompts U[256, 2048], 0-2 cached blocks,
    32/8/128, bs 256).  A step is attn_prefill_varlen_append: the store of
    the uncached suffix fused into the paged prefill, launched eagerly as the
    engine runs prefill steps.  The same step as two launches (kv_store, then
    attn_prefill_varlen) is timed in a second loop, with the store's own
    roofline."""
    wp = W.config3_prefill()
    flops = prefill_flops(wp)
    psets = [DeviceSet(wp, dev) for _ in range(args.sets)]
    psteps = args.prefill_steps or max(50, args.steps // 4)
    ms_pstep, _, pwin = timed_loop_eager(no_call, lambda s_: prefill_append_call(kvp, s_, wp),
                                         psets, psteps, args.warmup, world, call_events=False)
    _, ms_fused, _ = timed_loop_eager(no_call, lambda s_: prefill_append_call(kvp, s_, wp), psets,
                                      psteps, args.warmup, world)
    assert kvp.device_status() == 0, "device status after the timed prefill loop"
    ms_step2, ms_prefill, pwin2 = timed_loop_eager(lambda s_: store_call(kvp, s_),
                                                   lambda s_: prefill_call(kvp, s_, wp), psets, psteps,
                                                   args.warmup, world)
    ms_store = timed_loop_eager.last_store_ms
    assert kvp.device_status() == 0, "device status after the two-call prefill loop"
    flops_per_s, ms_pstep = aggregate(flops, ms_pstep, world)
    flops_per_s2, ms_step2 = aggregate(flops, ms_step2, world)
    tf_fused = flops / (ms_fused * 1e-3) / 1e12
    tf_prefill = flops / (ms_prefill * 1e-3) / 1e12
    # the suffix store: every new row's K and V read and written, plus slot_mapping
    n_new = int(wp.steps[0].store.slot_mapping.shape[0])
    store_bytes = n_new * (4 * wp.num_kv_heads * wp.head_dim * 2 + 4)
    store_gbs = store_bytes / (ms_store * 1e-3) / 1e9
    del psets
    return {"window": pwin, "window2": pwin2,
            "line": {"workload": wp.description, "value": round(flops_per_s / 1e12, 2),
                     "unit": "TFLOP/s", "ms_per_step": round(ms_pstep, 4), "steps": psteps,
                     "step": "attn_prefill_varlen_append: kv_store of the uncached suffix fused into the "
                             "paged prefill, launched eagerly as the engine runs prefill steps",
                     "frac_of_bf16_burst": round(flops_per_s / 1e12 / peaks["bf16_tflops"], 4),
                     "roofline": {"kernel": "attn_prefill_varlen_append (store + prefill)", "bound": "tensor",
                                  "achieved": round(tf_fused, 1), "peak": peaks["bf16_tflops"],
                                  "unit": "TFLOP/s", "frac": round(tf_fused / peaks["bf16_tflops"], 4),
                                  "traffic": traffic_for("prefill"), "algorithmic_flops": flops,
                                  "peak_source": peaks["source"] + " bf16 burst",
                                  "ms_per_launch": round(ms_fused, 5)},
                     "two_calls": {
                         "step": "kv_store of the uncached suffix, then attn_prefill_varlen (two launches)",
                         "value": round(flops_per_s2 / 1e12, 2), "unit": "TFLOP/s",
                         "ms_per_step": round(ms_step2, 4),
                         "roofline": {"kernel": "attn_prefill_varlen", "bound": "tensor",
                                      "achieved": round(tf_prefill, 1), "peak": peaks["bf16_tflops"],
                                      "unit": "TFLOP/s", "frac": round(tf_prefill / peaks["bf16_tflops"], 4),
                                      "algorithmic_flops": flops, "peak_source": peaks["source"] + " bf16 burst",
                                      "ms_per_launch": round(ms_prefill, 5)},
                         "store": {"workload": f"kv_store of the prefill step's {n_new} new rows "
                                               f"({wp.num_kv_heads}x{wp.head_dim} bf16 K and V each)",
                                   "ms_per_launch": round(ms_store, 5),
                                   "roofline": {"kernel": "kv_store", "bound": "hbm",
                                                "achieved": round(store_gbs, 1), "peak": peaks["hbm_gbs"],
                                                "unit": "GB/s",
                                                "frac": round(store_gbs / peaks["hbm_gbs"], 4),
                                                "traffic": traffic_for("kv_store"),
                                                "algorithmic_bytes": store_bytes,
                                                "peak_source": peaks["source"]}}}}}


def measure_mixed(args, kvp, W, dev, stream, world, peaks):
    """One engine step mixing chunked prefill and decode (4 prompt chunks,
    3772 tokens, + 128 decode rows, 32/8/128), launched eagerly over 2 input
    sets in rotation.  The step is attn_mixed_step: the chunks through the
    fused store + prefill on part of the SMs, the decode rows through the
    decode kernel (store fused) on the others (5/8 of the SMs by default),
    side by side; a short sweep of
    the decode rows' SM share, and the same step as one
    attn_prefill_varlen_append call (decode rows as q_len-1 sequences of the
    prefill kernel), are reported beside it."""
    import torch
    wm = W.mixed_step_workload()
    flops = prefill_flops(wm)
    m = wm.steps[0].attn.meta
    nd = 128
    # algorithmic bytes: K and V of every sequence's keys once per kv head, q read, out written,
    # the new rows read and stored
    kv_bytes = int(m.cu_seqlens_k[-1]) * wm.num_kv_heads * wm.head_dim * 2 * 2
    qo_bytes = int(m.cu_seqlens_q[-1]) * wm.num_heads * wm.head_dim * 2 * 2
    st_bytes = int(m.cu_seqlens_q[-1]) * (4 * wm.num_kv_heads * wm.head_dim * 2 + 4)
    nbytes = kv_bytes + qo_bytes + st_bytes
    msets = [DeviceSet(wm, dev) for _ in range(2)]
    ws = torch.empty(kvp.attn_decode_workspace_size(nd, wm.num_heads, wm.head_dim, m.max_seqlen_k,
                                                    wm.block_size), dtype=torch.uint8, device=dev)
    steps = max(50, min(400, args.steps // 10))

    def mixed(s_, dsms=0):
        kvp.attn_mixed_step(s_.q, s_.k, s_.v, s_.slots, s_.cu_q, s_.cu_k, s_.max_q, s_.max_k, s_.kc, s_.vc,
                            s_.bt, nd, decode_sms=dsms, softmax_scale=wm.scale, workspace=ws, out=s_.out)

    ms_step, _, win = timed_loop_eager(no_call, mixed, msets, steps, args.warmup, world, call_events=False)
    _, ms_call, _ = timed_loop_eager(no_call, mixed, msets, steps, args.warmup, world)
    sweep = {}
    for dsms in (76, 88, 96, 100):
        t, _, _ = timed_loop_eager(no_call, lambda s_: mixed(s_, dsms), msets, steps, 3, world,
                                   call_events=False)
        sweep[str(dsms)] = round(nbytes / (t * 1e-3) / 1e9, 1)
    ms_one, _, _ = timed_loop_eager(no_call, lambda s_: prefill_append_call(kvp, s_, wm), msets, steps,
                                    args.warmup, world, call_events=False)
    assert kvp.device_status() == 0, "device status after the mixed loops"
    fps, ms_step = aggregate(flops, ms_step, world)
    tf_call = flops / (ms_call * 1e-3) / 1e12
    gbs_call = nbytes / (ms_call * 1e-3) / 1e9
    del msets, ws
    return {"window": win, "steps": steps,
            "line": {"workload": wm.description, "value": round(nbytes / (ms_step * 1e-3) / 1e9, 1),
                     "unit": "GB/s", "ms_per_step": round(ms_step, 4), "steps": steps,
                     "step": "attn_mixed_step: chunks (store + prefill) beside the 128 decode rows "
                             "(decode, store fused) on 95 of the 152 SMs, one stream, chained by programmatic "
                             "dependent launches",
                     "roofline": {"kernel": "attn_mixed_step (store + prefill | decode)", "bound": "hbm",
                                  "achieved": round(gbs_call, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(gbs_call / peaks["hbm_gbs"], 4), "traffic": traffic_for("mixed"),
                                  "algorithmic_bytes": nbytes, "peak_source": peaks["source"],
                                  "ms_per_launch": round(ms_call, 5),
                                  "tensor": {"achieved_tflops": round(tf_call, 1),
                                             "frac_of_bf16_burst": round(tf_call / peaks["bf16_tflops"], 4),
                                             "algorithmic_flops": flops}},
                     "decode_sms_sweep_gbs": sweep,
                     "one_call": {"step": "attn_prefill_varlen_append over chunks and decode rows",
                                  "ms_per_step": round(ms_one, 4),
                                  "value": round(nbytes / (ms_one * 1e-3) / 1e9, 1), "unit": "GB/s",
                                  "frac_of_hbm": round(nbytes / (ms_one * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}}}


def measure_bucketed(args, kvp, W, dev, stream, world, peaks):
    """The engine's graph-replayed decode with batch-size buckets: a step of
    50 sequences (16/8/128, bs 256, ctx U[512, 4096], 2048-block pool) loads
    its metadata (slot_mapping, context_lens, block tables, packed for the
    bucket with its 14 padding rows: slot -1, context 0) in one copy from
    pinned host memory and replays the bucket-64 graph.  q, k and v sit in the
    graph's fixed buffers, where an engine's projections write them.  Value =
    algorithmic bytes of the 50 real sequences / step time.  A second loop
    times ``run`` with every input (q, k, v and metadata) copied from device
    tensors into the graph's buffers, as separate copies."""
    import torch
    from paged_kv_cache_125_gb300.graphs import DecodeGraphs
    g = torch.Generator().manual_seed(W.SEED_LENGTHS)
    ctx = torch.randint(512, 4097, (50,), generator=g).tolist()
    w = W.decode_workload("decode_b50_bucketed", ctx, 16, 8, 128, 256, 2048)
    kc, vc = w.new_cache(dev, poison=True)
    w.place_history(kc, vc)
    graphs = DecodeGraphs(kc, vc, 16, 16, max_bs=64, stream=stream)
    st, a = w.steps[0].store, w.steps[0].attn
    b = len(ctx)
    ins = [a.q.to(dev), st.k.to(dev), st.v.to(dev), st.slot_mapping.to(dev),
           a.meta.block_tables.to(dev), a.meta.context_lens.to(dev)]
    graphs.q[:b].copy_(ins[0])
    graphs.k[:b].copy_(ins[1])
    graphs.v[:b].copy_(ins[2])
    packed = graphs.pack(b, st.slot_mapping, a.meta.block_tables, a.meta.context_lens,
                         out=torch.empty((graphs.meta.numel(),), dtype=torch.int32, pin_memory=True))
    store_b, dec_b = decode_bytes(w)
    steps = max(100, min(2000, args.steps // 5))

    def loop(fn, n):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        barrier(world)
        w0 = time.perf_counter()
        t0.record()
        for _ in range(n):
            fn()
        t1.record()
        torch.cuda.synchronize()
        w1 = time.perf_counter()
        barrier(world)
        return t0.elapsed_time(t1) / n, (w0, w1)

    for _ in range(max(3, args.warmup)):
        graphs.run_packed(b, packed)
    ms, win = loop(lambda: graphs.run_packed(b, packed), steps)
    assert kvp.device_status() == 0, "device status after the bucketed loop"
    for _ in range(max(3, args.warmup)):
        graphs.run(*ins)
    ms_copies, _ = loop(lambda: graphs.run(*ins), steps)
    assert kvp.device_status() == 0, "device status after the bucketed loop (run)"
    bps, ms = aggregate(store_b + dec_b, ms, world)
    bps_c, ms_copies = aggregate(store_b + dec_b, ms_copies, world)
    del graphs, kc, vc
    return {"window": win, "steps": 2 * steps,
            "line": {"workload": "decode B50 padded to the bucket-64 graph, 16/8/128 bs256 NB2048 "
                                 "ctx U[512,4096]", "value": round(bps / 1e9, 2), "unit": "GB/s",
                     "ms_per_step": round(ms, 4), "steps": steps,
                     "step": "one copy of the packed metadata (pinned host -> device) + replay "
                             "(attn_decode_paged_append); q/k/v in the graph's buffers",
                     "frac_of_hbm": round(bps / 1e9 / peaks["hbm_gbs"], 4),
                     "inputs_copied": {"step": "q, k, v, slot_mapping, block_tables, context_lens "
                                               "copied device -> graph buffers (6 copies, 2 fills) "
                                               "+ replay", "value": round(bps_c / 1e9, 2),
                                       "unit": "GB/s", "ms_per_step": round(ms_copies, 4)}}}


def measure_decode_large(args, kvp, W, dev, stream, world, peaks):
    """The bandwidth sweep configuration: 512 sequences, Qwen3-8B heads
    (32/8/128), bs 256, contexts 50% U[128, 1024] + 50% U[4096, 8192], over a
    143,051-block pool (150 GB of K+V, unreferenced blocks NaN).  One input set
    (the step reads ~7 GB, 55x the L2); store + decode graphs as in the main
    line."""
    import torch
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info(dev)
    blocks = args.b512_blocks or W.CONFIG4_POOL_BLOCKS
    need = blocks * 2 * 256 * 8 * 128 * 2 * 1.1
    if free < need:
        return {"window": None, "steps": 0,
                "line": {"skipped": f"needs ~{need / 1e9:.0f} GB free device memory, "
                                    f"{free / 1e9:.0f} GB free"}}
    w = W.config4_decode(num_blocks=blocks, batch=args.b512_batch, device=dev)
    store_b, dec_b = decode_bytes(w)
    ds = DeviceSet(w, dev)
    m = w.steps[0].attn.meta
    ws = torch.empty(kvp.attn_decode_workspace_size(args.b512_batch, 32, 128, m.max_context_len, 256),
                     dtype=torch.uint8, device=dev)
    ag = capture(lambda s_: append_call(kvp, s_, w, ws), [ds], stream)
    steps = max(10, min(100, args.steps // 100))
    ms_step, ms_dec, win = timed_loop_single(ag, steps, max(3, args.warmup // 4), world)
    assert kvp.device_status() == 0, "device status after the large decode loop"
    bps, ms_step = aggregate(store_b + dec_b, ms_step, world)
    achieved = (store_b + dec_b) / (ms_dec * 1e-3) / 1e9
    del ag, ds, ws
    torch.cuda.empty_cache()
    return {"window": win, "steps": steps,
            "line": {"workload": w.description, "value": round(bps / 1e9, 2), "unit": "GB/s",
                     "ms_per_step": round(ms_step, 4), "steps": steps,
                     "step": "attn_decode_paged_append (kv_store of 512 new rows fused)",
                     "roofline": {"kernel": "attn_decode_paged_append (store + split + merge)",
                                  "bound": "hbm",
                                  "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(achieved / peaks["hbm_gbs"], 4),
                                  "traffic": traffic_for("decode_b512") if args.b512_batch == 512 else None,
                                  "algorithmic_bytes": store_b + dec_b, "peak_source": peaks["source"],
                                  "ms_per_launch": round(ms_dec, 5)}}}


def measure_decode_group8(args, kvp, W, dev, stream, world, peaks):
    """Decode with eight query heads per kv head at head_dim 128 (64/8/128):
    the decode B64 batch (64 sequences, ctx U[512, 4096], bs 256, 2048-block
    pool) with that attention shape, store fused, 2 input sets in rotation
    (2.3 GB of pools)."""
    import torch
    ctx = torch.randint(512, 4097, (64,), generator=W.generator(W.SEED_LENGTHS)).tolist()
    w = W.decode_workload("decode_b64_g8", ctx, 64, 8, 128, 256, 2048,
                          description="decode: B64 64/8/128 bs256 NB2048 ctx U[512,4096]")
    store_b, dec_b = decode_bytes(w)
    sets = [DeviceSet(w, dev) for _ in range(2)]
    ws = torch.empty(kvp.attn_decode_workspace_size(64, 64, 128, w.steps[0].attn.meta.max_context_len, 256),
                     dtype=torch.uint8, device=dev)
    graphs = capture(lambda s_: append_call(kvp, s_, w, ws), sets, stream)
    steps = max(20, min(200, args.steps // 25))
    ms_step, ms_call, win = timed_loop_single(graphs, steps, max(3, args.warmup // 4), world)
    assert kvp.device_status() == 0, "device status after the group-8 decode loop"
    achieved = (store_b + dec_b) / (ms_call * 1e-3) / 1e9
    del graphs, sets, ws
    torch.cuda.empty_cache()
    return {"window": win, "steps": steps,
            "line": {"workload": w.description, "ms_per_step": round(ms_step, 4), "steps": steps,
                     "step": "attn_decode_paged_append (store fused)",
                     "roofline": {"kernel": "attn_decode_paged_append (store + split + merge)",
                                  "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                                  "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                                  "traffic": traffic_for("decode_group8"), "algorithmic_bytes": store_b + dec_b,
                                  "peak_source": peaks["source"], "ms_per_launch": round(ms_call, 5)}}}


def measure_trace(args, kvp, dev, stream, world, peaks):
    """Engine-trace replay: 256 requests (prompts and outputs U[100, 1024]),
    scheduled by the native scheduler (prefill first, max 512 seqs / 16384
    tokens per step, 768 blocks of 256 tokens), every step running kv_store +
    prefill or decode attention on all 28 layers of a Qwen3-0.6B attention
    shape (16/8/128), with per-layer q/k/v drawn on the device.  The step loop
    is ``EngineReplay`` (the one the GPU trace test checks against the
    oracle): prefill steps are launched eagerly; decode steps replay one
    28-layer graph per batch-size bucket, as the pages' engine does.
    Aggregate GB/s over the decode steps (algorithmic bytes) and TFLOP/s over
    the prefill steps (causal FLOPs), each timed by an event pair around
    ``launch`` (for decode: the copy of the step's packed metadata into the
    graph's buffer and the replay).  Prefill steps are also broken down by
    their query tokens, with the host's issue time per layer call (measured
    with an empty launch queue)."""
    import torch
    from paged_kv_cache_125_gb300 import engine_trace as E
    from paged_kv_cache_125_gb300.engine_replay import (EngineReplay, decode_bytes, prefill_flops,
                                                        prefill_layer_bytes)
    layers, hq, hkv, d, bs, nb = 28, 16, 8, 128, 256, 768
    torch.cuda.empty_cache()
    reqs = E.make_requests(256, (100, 1024), (100, 1024))
    eng = EngineReplay(reqs, layers, hq, hkv, d, bs, nb, 512, 16384, dev, stream=stream)
    gq = torch.Generator(device=dev).manual_seed(5)
    recs = []
    w0 = time.perf_counter()
    while not eng.done():
        st = eng.schedule()
        n = st.num_new
        if st.is_prefill:
            q = torch.randn((layers, n, hq, d), generator=gq, device=dev).to(torch.bfloat16)
            k = torch.randn((layers, n, hkv, d), generator=gq, device=dev).to(torch.bfloat16)
            v = torch.randn((layers, n, hkv, d), generator=gq, device=dev).to(torch.bfloat16)
            work = prefill_flops(st.meta, d, hq)
            pbytes = prefill_layer_bytes(st.meta, hq, hkv, d)
        else:  # every layer's new rows, straight into the graph's buffers
            q, k, v = eng.decode_inputs(st)
            q.copy_(torch.randn(q.shape, generator=gq, device=dev))
            k.copy_(torch.randn(k.shape, generator=gq, device=dev))
            v.copy_(torch.randn(v.shape, generator=gq, device=dev))
            work = decode_bytes(st.meta, n, hq, hkv, d, bs)
            pbytes = 0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if st.is_prefill:
            # Drain the launch queue (the host runs steps ahead of the device,
            # and a full queue blocks launches), then keep the device busy for
            # ~100 us outside the event pair while the host issues the layers:
            # host_us is then the issue time alone, and the events see no
            # start-up gap.
            torch.cuda.synchronize()
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(200_000)
        a.record()
        h0 = time.perf_counter()
        eng.launch(st, q, k, v)
        host_us = (time.perf_counter() - h0) * 1e6
        b.record()
        recs.append((st.is_prefill, work * layers, a, b, n, len(st.seq_ids), host_us, pbytes * layers))
        eng.commit(st, [(7 * i + n) % 151936 for i in st.seq_ids])
        del q, k, v
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    assert kvp.device_status() == 0, "device status after the trace replay"
    dec_ms = sum(a.elapsed_time(b) for p_, _, a, b, *_ in recs if not p_)
    pre_ms = sum(a.elapsed_time(b) for p_, _, a, b, *_ in recs if p_)
    dec_work = sum(w_ for p_, w_, *_ in recs if not p_)
    pre_work = sum(w_ for p_, w_, *_ in recs if p_)
    n_dec = sum(1 for r in recs if not r[0])
    # prefill steps by query tokens; each step's roofline time is the larger of its algorithmic
    # bytes at the measured copy bandwidth and its FLOPs at the measured bf16 burst peak
    groups = {}
    roof_ms = 0.0
    for p_, w_, a, b, n, ns, host_us, pb in recs:
        if not p_:
            continue
        key = ">=8192 tokens" if n >= 8192 else ("1024-8191 tokens" if n >= 1024 else "<1024 tokens")
        g = groups.setdefault(key, {"steps": 0, "tokens": 0, "seqs": 0, "ms": 0.0, "tflop": 0.0,
                                    "gbytes": 0.0, "roof_ms": 0.0, "host_ms": 0.0})
        r_ms = max(pb / (peaks["hbm_gbs"] * 1e9), w_ / (peaks["bf16_tflops"] * 1e12)) * 1e3
        roof_ms += r_ms
        g["steps"] += 1
        g["tokens"] += n
        g["seqs"] += ns
        g["ms"] += a.elapsed_time(b)
        g["tflop"] += w_ / 1e12
        g["gbytes"] += pb / 1e9
        g["roof_ms"] += r_ms
        g["host_ms"] += host_us / 1e3
    for g in groups.values():
        g["ms"] = round(g["ms"], 3)
        g["tflop"] = round(g["tflop"], 4)
        g["gbytes"] = round(g["gbytes"], 3)
        g["us_per_layer_call"] = round(g["ms"] * 1e3 / (g["steps"] * layers), 2)
        g["roofline_us_per_layer_call"] = round(g["roof_ms"] * 1e3 / (g["steps"] * layers), 2)
        g["frac_of_roofline"] = round(g.pop("roof_ms") / g["ms"], 4)
        g["host_us_per_layer_call"] = round(g.pop("host_ms") * 1e3 / (g["steps"] * layers), 2)
        g["tflops"] = round(g["tflop"] / (g["ms"] * 1e-3), 1)
    preempt = eng.num_preemptions
    del eng
    torch.cuda.empty_cache()
    dec_gbs = dec_work / (dec_ms * 1e-3) / 1e9
    pre_tf = pre_work / (pre_ms * 1e-3) / 1e12
    return {"window": (w0, w1), "launches": 2 * layers * len(recs),
            "line": {"workload": "engine trace: 256 requests, prompts/outputs U[100,1024], 28 layers "
                                 "16/8/128, bs 256, 768 blocks, native scheduler",
                     "steps": len(recs), "decode_steps": n_dec, "prefill_steps": len(recs) - n_dec,
                     "preemptions": preempt,
                     "decode": {"value": round(dec_gbs, 2), "unit": "GB/s", "ms": round(dec_ms, 2),
                                "frac_of_hbm": round(dec_gbs / peaks["hbm_gbs"], 4)},
                     "prefill": {"value": round(pre_tf, 2), "unit": "TFLOP/s", "ms": round(pre_ms, 2),
                                 "frac_of_bf16_burst": round(pre_tf / peaks["bf16_tflops"], 4),
                                 "frac_of_roofline": round(roof_ms / pre_ms, 4),
                                 "roofline": "per step: max(algorithmic bytes / measured copy bandwidth, "
                                             "causal FLOPs / measured bf16 burst peak); bytes per layer "
                                             "call: q, the new K/V rows read and stored, the output, and "
                                             "the cached prefix's K/V",
                                 "by_query_tokens": groups},
                     "how": "EngineReplay: event pair around each step's launch of 28 layers (prefill: "
                            "attn_prefill_varlen_append per layer, eager; decode: one copy of the "
                            "packed metadata from pinned memory + one 28-layer graph replay of "
                            "attn_decode_paged_append per bucket); per-layer inputs generated on the "
                            "device before each step"}}


def measure_scheduler():
    """Host step loop of the engine-trace configuration (256 requests, 768
    blocks of 256 tokens, max 512 seqs / 16384 tokens per step, 1371 steps):
    schedule + metadata + postprocess per step, native C++ scheduler (through
    its C ABI) against the Python replica of the same policy."""
    from paged_kv_cache_125_gb300 import engine_trace as E
    from paged_kv_cache_125_gb300.scheduler import NativeScheduler
    reqs = E.make_requests(256, (100, 1024), (100, 1024))

    def py_loop():
        sch = E.Scheduler(512, 16384, 768, 256)
        for i, (t, o) in enumerate(reqs):
            sch.submit(E.Request(i, t, o, 256))
        n = 0
        while not sch.done():
            seqs, pre = sch.next_batch()
            E.step_metadata(seqs, pre, 256)
            sch.commit(seqs, [E.synthetic_token(x.rid, len(x)) for x in seqs])
            n += 1
        return n

    def native_loop():
        sch = NativeScheduler(768, 256, 512, 16384)
        for i, (t, o) in enumerate(reqs):
            sch.add(i, t, o)
        n = 0
        while not sch.is_finished():
            ids, _, _ = sch.step()
            sch.postprocess([(7 * i + n) % 151936 for i in ids])
            n += 1
        return n

    # Best of three whole runs each: the host is shared, one run can be slowed
    # by other work on its cores.
    out = {}
    for name, f in (("native", native_loop), ("python_replica", py_loop)):
        best = float("inf")
        for _ in range(3):
            t0 = time.perf_counter()
            n = f()
            best = min(best, (time.perf_counter() - t0) / n * 1e6)
        out[name] = round(best, 1)
        out["steps"] = n
    return {"workload": "engine trace: 256 requests, 768 blocks x 256 tokens, 512 seqs / 16384 tokens per step",
            "unit": "us/step (host: schedule + metadata + postprocess), best of 3 runs",
            "native": out["native"], "python_replica": out["python_replica"], "steps": out["steps"]}


def measure_copy_blocks(args, kvp, dev, stream, world, peaks):
    """Copy-on-write block copies (page 3, "场景优化1：Parallel Memory Shared"):
    one call copies 64 (src, dst) block pairs in all 56 planes of a 28-layer
    cache of 512 KiB blocks (Qwen3-0.6B shape, bs 256) = 3.76 GB of traffic;
    every byte read once and written once."""
    import torch
    layers, nb, bs, hkv, d, pairs = 28, 160, 256, 8, 128, 64
    cache = torch.zeros((2, layers, nb, bs, hkv, d), dtype=torch.bfloat16, device=dev)
    g = torch.Generator().manual_seed(2)
    perm = torch.randperm(nb, generator=g)
    dst = perm[:pairs]
    src = perm[pairs:][torch.randint(0, nb - pairs, (pairs,), generator=g)]
    mapping = torch.stack([src, dst], dim=1).to(torch.int32).to(dev)
    block_bytes = bs * hkv * d * 2
    step_bytes = 2 * pairs * 2 * layers * block_bytes
    steps = max(10, min(50, args.steps // 100))
    for _ in range(3):
        kvp.kv_copy_blocks(cache, mapping)
    torch.cuda.synchronize()
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    w0 = time.perf_counter()
    for a, b in evs:
        a.record()
        kvp.kv_copy_blocks(cache, mapping)
        b.record()
    torch.cuda.synchronize()
    w1 = time.perf_counter()
    barrier(world)
    assert kvp.device_status() == 0, "device status after the copy loop"
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    bps, ms = aggregate(step_bytes, ms, world)
    achieved = step_bytes / (ms * 1e-3) / 1e9
    del cache
    return {"window": (w0, w1),
            "line": {"workload": f"copy-on-write: {pairs} block pairs x {2 * layers} planes "
                                 f"(28 layers K+V, bs {bs}, 8x128, 512 KiB blocks), pool {nb} blocks",
                     "value": round(bps / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
                     "steps": steps,
                     "roofline": {"kernel": "kv_copy_blocks", "bound": "hbm", "achieved": round(achieved, 1),
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic_for("copy_blocks"),
                                  "algorithmic_bytes": step_bytes, "peak_source": peaks["source"],
                                  "ms_per_launch": round(ms, 5)}}}


def run_ours(args, rank, world, local):
    import torch
    import paged_kv_cache_125_gb300 as kvp
    from paged_kv_cache_125_gb300 import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    sampler.start()
    time.sleep(0.3)
    windows = []
    dec = pre = None
    single = {"decode_b512": lambda: measure_decode_large(args, kvp, W, dev, stream, world, peaks),
              "decode_group8": lambda: measure_decode_group8(args, kvp, W, dev, stream, world, peaks),
              "mixed": lambda: measure_mixed(args, kvp, W, dev, stream, world, peaks),
              "copy_blocks": lambda: measure_copy_blocks(args, kvp, dev, stream, world, peaks),
              "decode_bucketed": lambda: measure_bucketed(args, kvp, W, dev, stream, world, peaks),
              "engine_trace": lambda: measure_trace(args, kvp, dev, stream, world, peaks)}
    if args.only in single:  # profiling run of one line only
        r = single[args.only]()
        clocks = sampler.stop([r["window"]] if r["window"] else [])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "only": args.only, "clocks": clocks,
                              args.only: r["line"]}), flush=True)
        return
    if args.only != "prefill":
        dec = measure_decode(args, kvp, W, dev, stream, world, peaks)
        windows += [dec["window"], dec["uwindow"]]
    if args.only != "decode" and not args.no_prefill:
        pre = measure_prefill(args, kvp, W, dev, stream, world, peaks)
        windows += [pre["window"], pre["window2"]]
    mx = None
    if args.only is None and not args.no_prefill:
        mx = measure_mixed(args, kvp, W, dev, stream, world, peaks)
        windows.append(mx["window"])
    bk = None
    if args.only is None:
        bk = measure_bucketed(args, kvp, W, dev, stream, world, peaks)
        windows.append(bk["window"])
    g8 = None
    if args.only is None:
        g8 = measure_decode_group8(args, kvp, W, dev, stream, world, peaks)
        windows.append(g8["window"])
    cb = None
    if args.only is None and not args.no_copy_blocks:
        cb = measure_copy_blocks(args, kvp, dev, stream, world, peaks)
        windows.append(cb["window"])
    tr = None
    if args.only is None and not args.no_trace:
        tr = measure_trace(args, kvp, dev, stream, world, peaks)
        windows.append(tr["window"])
    dl = None
    if args.only is None and not args.no_large:
        dl = measure_decode_large(args, kvp, W, dev, stream, world, peaks)
        if dl["window"] is not None:
            windows.append(dl["window"])
    time.sleep(0.1)
    clocks = sampler.stop(windows)

    cpu = None
    if dec is not None and rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sec, reps, cores = oracle_decode_rate(dec["w"], min_seconds=8.0)
        cpu = {"value": round(rate, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"full decode step (store + decode, 64 sequences) x {reps}, {sec:.2f} s each"}
    if rank != 0:
        return
    if dec is None:  # profiling run of the prefill half only
        print(json.dumps({"metric": METRIC, "only": "prefill", "clocks": clocks, "prefill": pre["line"]}),
              flush=True)
        return
    w = dec["w"]
    line = {"metric": METRIC, "value": round(dec["value"], 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dec["ms_step"], 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": bench_config(w, args.sets),
            "setup": {"step": "attn_decode_paged_append: kv_store of the 64 new rows fused into the "
                              "paged decode (split + merge)",
                      "global_batch": 64 * world,
                      "graph": "each step is one CUDA graph replay"},
            "parallelism": f"replicas x{world}",
            "roofline": dec["roofline"], "cpu_baseline": cpu, "e2e": dec["e2e"],
            "unfused": dec["unfused"],
            "gpu_launches": 2 * args.steps + 3 * args.steps
                            + (0 if pre is None else 6 * pre["line"]["steps"])
                            + (0 if cb is None else cb["line"]["steps"])
                            + (0 if mx is None else 26 * mx["steps"])
                            + (0 if bk is None else 2 * bk["steps"])
                            + (0 if g8 is None else 2 * g8["steps"])
                            + (0 if dl is None else 2 * dl["steps"])
                            + (0 if tr is None else tr["launches"]),
            "gpu_launches_by_region": {"decode": {"decode_split": args.steps,
                                                  "decode_merge": args.steps},
                                       "decode_unfused": {"kv_store": args.steps,
                                                          "decode_split": args.steps,
                                                          "decode_merge": args.steps},
                                       "prefill": None if pre is None else
                                       {"kv_store_narrow (fused calls, 2 loops)": 2 * pre["line"]["steps"],
                                        "prefill (fused calls, 2 loops)": 2 * pre["line"]["steps"],
                                        "kv_store (two-call loop)": pre["line"]["steps"],
                                        "prefill (two-call loop)": pre["line"]["steps"]},
                                       "copy_blocks": None if cb is None else
                                       {"kv_copy_blocks": cb["line"]["steps"]},
                                       "mixed": None if mx is None else
                                       {"attn_mixed_step: store, prefill, split, merge (6 loops)":
                                        24 * mx["steps"],
                                        "attn_prefill_varlen_append: store, prefill (1 loop)": 2 * mx["steps"]},
                                       "engine_trace": None if tr is None else {"all": tr["launches"]},
                                       "decode_b512": None if dl is None or not dl["steps"] else
                                       {"decode_split": dl["steps"], "decode_merge": dl["steps"]},
                                       "decode_bucketed": None if bk is None else
                                       {"decode_split": bk["steps"], "decode_merge": bk["steps"]},
                                       "decode_group8": None if g8 is None else
                                       {"decode_split": g8["steps"], "decode_merge": g8["steps"]}},
            "clocks": clocks,
            "prefill": None if pre is None else pre["line"],
            "mixed": None if mx is None else mx["line"],
            "scheduler": measure_scheduler() if args.only is None else None,
            "decode_bucketed": None if bk is None else bk["line"],
            "decode_b512": None if dl is None else dl["line"],
            "decode_group8": None if g8 is None else g8["line"],
            "engine_trace": None if tr is None else tr["line"],
            "copy_blocks": None if cb is None else cb["line"]}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_info()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
