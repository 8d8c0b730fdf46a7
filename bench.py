#!/usr/bin/env python
"""Benchmark of paged GQA decode attention on GB300.

Metric: paged decode attention microseconds per call and achieved HBM GB/s
(K + V + q + out bytes over the call's time) as a fraction of the measured
HBM peak, on one GPU.  One "step" is one ``pda_decode`` call over the whole
batch (one kernel launch: the split pieces of a unit merge inside it).
Default workload: the 8B-style batch (B=32, Hq=32, Hkv=8, D=128, block 16,
4096 tokens each; 537 MB moved per call).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 8b|1b|wide|ragged|tiny] [--block-size BS]
                  [--q-len Q] [--multi-form mma|tc] [--layout paged|contiguous]
                  [--tiles T] [--no-graph] [--no-e2e] [--no-cpu-baseline] [--no-others] [--quick]

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(the fp64 definition) on this host's cores instead of the GPU path.
``--q-len`` decodes Q causal queries per sequence, ``--layout contiguous``
the same cache as [B, S, Hkv, D], ``--tiles`` through the tiled lifecycle.
The default run (the 8B batch, paged, one query) also times the other four
named workloads (tiny, 1b, wide, ragged) the same way and adds them to its
line as ``other_configs``; the headline value stays the 8B batch.

Timing: CUDA events on the launching stream around exactly K back-to-back
calls after W warm-up calls; inputs are larger than L2 and rotate between
copies at distinct addresses.  The K calls are captured once in a CUDA graph
and replayed (the host's per-call launch cost would otherwise bound the small
workloads); the same calls launched one by one are timed too (``loop``).  A
second pass records events around the kernel of each call (which stops the
next call's early launch): an isolated-launch time, reported beside the
roofline, whose achieved rate uses the graph-replayed per-launch time (a
decode call is one kernel launch).  ``e2e`` repeats the calls with the inputs copied from pinned
host memory and the output copied back every step.
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

METRIC = "paged decode attn μs/call and KV GB/s as % of GB300 HBM peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="8b")
    ap.add_argument("--block-size", type=int, default=0,
                    help="redraw the workload with this block size (e.g. 1 for token pages)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="causal queries per sequence (pda_decode_multi) instead of one")
    ap.add_argument("--multi-form", choices=["mma", "tc"], default="mma",
                    help="with --q-len: launch rows of 17-32 q rows on the mma.sync row form "
                         "(the default) or the tcgen05 one")
    ap.add_argument("--tiles", type=int, default=0,
                    help="decode with the tiled lifecycle instead: begin_step, this many "
                         "step_tile calls (each 1/T of every sequence's blocks), finalize")
    ap.add_argument("--layout", choices=["paged", "contiguous"], default="paged",
                    help="contiguous: the same cache copied to [B, S, Hkv, D] and decoded "
                         "with pda_decode_contiguous")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the K calls launched one by one from Python instead of replaying "
                         "them from a CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="skip timing the other named workloads (tiny, 1b, wide, ragged) that "
                         "the default run adds to its line as other_configs")
    ap.add_argument("--quick", action="store_true",
                    help="only the W + K calls: no clock padding, kernel-timing pass, e2e or "
                         "CPU baseline (for profiler captures)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, device) -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The files the decode kernels are compiled from (host-only files
# such as pda_api.cu do not change the kernels' traffic).
KERNEL_SOURCES = ("pda_kernels.cuh", "pda_ptx.cuh", "pda_params.h", "pda_plan.h",
                  "pda_kernels_d64.cu", "pda_kernels_d128.cu", "pda_kernels_d256.cu")


def kernel_source_hash() -> str:
    """Hash of the kernel sources with // comments, trailing blanks and empty
    lines dropped, so that a change to comments alone keeps the record."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_gqa_decode_05_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload_key: str):
    """Per-launch DRAM bytes of the split kernel from the committed ncu summary,
    or None when the kernel source changed since it was captured."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = d.get("workloads", {}).get(workload_key)
    return None if entry is None else float(entry["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_timing(w, budget_s: float = 10.0):
    """Times the oracle as it stands on all host cores over a bounded sample of
    the workload's (b, h) outputs (all of them when that fits the budget)."""
    import numpy as np
    import oracle
    orc = oracle.load()
    threads = oracle.host_threads()
    total_pairs = w.B * w.Hq
    args = (w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens)
    kw = dict(Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size, n_threads=threads)
    rng = np.random.default_rng(0)
    # probe with a small sample to size the bounded one
    probe = rng.choice(total_pairs, size=min(total_pairs, max(threads, 16)), replace=False)
    probe_pairs = np.stack([probe // w.Hq, probe % w.Hq], axis=1).astype(np.int32)
    t = time.perf_counter()
    orc.decode(*args, **kw, pairs=probe_pairs)
    per_pair = (time.perf_counter() - t) / len(probe)
    n = int(min(total_pairs, max(len(probe), budget_s / max(per_pair, 1e-9))))
    if n >= total_pairs:
        pairs, desc = None, f"all {total_pairs} (b, q-head) outputs of the workload"
    else:
        pick = np.sort(rng.choice(total_pairs, size=n, replace=False))
        pairs = np.stack([pick // w.Hq, pick % w.Hq], axis=1).astype(np.int32)
        desc = f"{n} of {total_pairs} (b, q-head) outputs drawn uniformly (seed 0)"
    reps, elapsed = 0, 0.0
    while reps < 1 or (elapsed < budget_s and reps < 3):
        t = time.perf_counter()
        orc.decode(*args, **kw, pairs=pairs)
        elapsed += time.perf_counter() - t
        reps += 1
    frac = (n if pairs is not None else total_pairs) / total_pairs
    sec_per_call = elapsed / reps / frac  # scaled to the whole workload
    gbs = w.algorithmic_bytes() / sec_per_call / 1e9
    # the same oracle on one thread, over a smaller sample of the same outputs
    n1 = int(min(total_pairs, max(1, budget_s / 4 / max(per_pair * threads, 1e-9))))
    pick1 = np.sort(rng.choice(total_pairs, size=n1, replace=False))
    pairs1 = np.stack([pick1 // w.Hq, pick1 % w.Hq], axis=1).astype(np.int32)
    t = time.perf_counter()
    orc.decode(*args, **{**kw, "n_threads": 1}, pairs=pairs1)
    sec1 = (time.perf_counter() - t) * total_pairs / n1
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{desc}; fp64 C oracle, {reps} repetition(s), scaled to the full call",
            "sec_per_call": sec_per_call,
            "single_thread": {"value": w.algorithmic_bytes() / sec1 / 1e9, "unit": "GB/s",
                              "sec_per_call": sec1,
                              "sample": f"{n1} of {total_pairs} (b, q-head) outputs, one thread, "
                                        "scaled to the full call"}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_gqa_decode_05_gb300 import workloads
    w = workloads.WORKLOADS[args.workload]()
    cb = cpu_oracle_timing(w, budget_s=10.0)
    line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": cb["sec_per_call"] * 1e3, "us_per_call": cb["sec_per_call"] * 1e6,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 inputs)",
            "config": {**w.describe(), "workload": w.name, "kv_layout": args.layout,
                   "q_len": args.q_len, "runs_on": "host CPU cores"},
            "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                "single_thread")},
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


OTHER_CONFIGS = ("tiny", "1b", "wide", "ragged")


def time_other_config(name: str, dev, steps: int, warmup: int, peak: float):
    """One of the other named decode workloads at its own shape, timed like the
    headline: calls replayed from a CUDA graph with inputs larger than L2
    rotated between copies, the split kernel alone with CUDA events around it,
    and the L2-warm figure where the inputs fit in L2."""
    import numpy as np
    import torch

    import paged_gqa_decode_05_gb300 as pda
    from paged_gqa_decode_05_gb300 import workloads

    w = workloads.WORKLOADS[name]()
    nbytes = w.algorithmic_bytes()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 2 ** 20))
    input_bytes = w.q.nbytes + w.k_pool.nbytes + w.v_pool.nbytes + w.block_table.nbytes + \
        w.seq_lens.nbytes
    n_sets = max(2, math.ceil(3 * l2 / max(input_bytes, 1)))

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    host = {"q": w.q, "k_pool": w.k_pool, "v_pool": w.v_pool, "block_table": w.block_table,
            "seq_lens": w.seq_lens}
    sets = [{k: to_dev(v) for k, v in host.items()} for _ in range(n_sets)]
    outs = [torch.empty(tuple(sets[0]["q"].shape), device=dev, dtype=torch.bfloat16)
            for _ in range(n_sets)]
    ctx = pda.Context(max_seqs=w.B, num_q_heads=w.Hq, num_kv_heads=w.Hkv, head_dim=w.D,
                      block_size=w.block_size)
    stream = torch.cuda.current_stream()
    counter = [0]

    def step(s=None, o=None):
        if s is None:
            i = counter[0]
            counter[0] += 1
            s, o = sets[i % n_sets], outs[i % n_sets]
        ctx.decode(s["q"], s["k_pool"], s["v_pool"], s["block_table"], s["seq_lens"], out=o)

    def graph_us(fn):
        for _ in range(max(3, warmup)):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(steps):
                    fn()
        stream.wait_stream(cap)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / steps

    us = graph_us(step)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    for k in range(steps):
        for e in evs[k]:
            e.record(stream)
        ctx.set_timing_events(*evs[k])
        step()
    ctx.set_timing_events(None, None, None)
    torch.cuda.synchronize()
    split_us = statistics.mean(a.elapsed_time(b) for a, b, _ in evs) * 1e3
    if ctx.read_device_errors() != 0:
        raise RuntimeError(f"device error flags set while timing {name}")
    r = {"workload": w.name, "algorithmic_bytes_per_call": nbytes, "us_per_call": us,
         "GB/s": nbytes / (us * 1e-6) / 1e9, "frac": nbytes / (us * 1e-6) / 1e9 / peak,
         "split_us": split_us, "split_GB/s": nbytes / (split_us * 1e-6) / 1e9,
         "split_frac": nbytes / (split_us * 1e-6) / 1e9 / peak, "steps": steps,
         "l2": f"{n_sets} input sets of {input_bytes / 1e6:.1f} MB rotated"}
    if input_bytes < l2 // 2:
        warm_us = graph_us(lambda: step(sets[0], outs[0]))
        r["l2_warm"] = {"us_per_call": warm_us, "GB/s": nbytes / (warm_us * 1e-6) / 1e9,
                        "note": "one input set reused every call (labelled; not the metric)"}
    ctx.close()
    del sets, outs
    torch.cuda.empty_cache()
    return r


def run_ours(args):
    import numpy as np
    import torch

    import paged_gqa_decode_05_gb300 as pda
    from paged_gqa_decode_05_gb300 import workloads

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    w = workloads.WORKLOADS[args.workload]()
    if args.block_size:
        w = workloads.with_block_size(w, args.block_size)
    if args.q_len > 1:
        w.q = workloads.multi_queries(w, args.q_len)
    # K+V of valid tokens once, q in and out (q_len rows each)
    bytes_per_call = w.algorithmic_bytes() + (args.q_len - 1) * 2 * w.B * w.Hq * w.D * 2
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 129 * 2 ** 20))
    input_bytes = (w.q.nbytes + w.k_pool.nbytes + w.v_pool.nbytes + w.block_table.nbytes
                   + w.seq_lens.nbytes)
    n_sets = max(2, math.ceil(3 * l2 / max(input_bytes, 1)))

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    if args.layout == "contiguous":
        k_c, v_c = workloads.contiguous_kv(w)
        host = {"q": w.q, "k_pool": k_c, "v_pool": v_c, "block_table": w.block_table,
                "seq_lens": w.seq_lens}
    else:
        host = {"q": w.q, "k_pool": w.k_pool, "v_pool": w.v_pool, "block_table": w.block_table,
                "seq_lens": w.seq_lens}
    sets = [{k: to_dev(v) for k, v in host.items()} for _ in range(n_sets)]
    outs = [torch.empty(tuple(sets[0]["q"].shape), device=dev, dtype=torch.bfloat16)
            for _ in range(n_sets)]
    tiles = []
    tile_cap = 64
    if args.tiles > 0:
        # tile i holds blocks [i*cap, (i+1)*cap) of every sequence (fewer at the end)
        nbs = -(-w.seq_lens.astype(np.int64) // w.block_size)
        tile_cap = max(1, int(-(-int(nbs.max()) // args.tiles)))
        for i in range(args.tiles):
            blocks = np.zeros((w.B, tile_cap), dtype=np.int32)
            counts = np.zeros(w.B, dtype=np.int32)
            last = np.full(w.B, w.block_size, dtype=np.int32)
            for b in range(w.B):
                lo, hi = min(i * tile_cap, int(nbs[b])), min((i + 1) * tile_cap, int(nbs[b]))
                blocks[b, :hi - lo] = w.block_table[b, lo:hi]
                counts[b] = hi - lo
                if hi == nbs[b] and hi > lo:
                    last[b] = int(w.seq_lens[b]) - (hi - 1) * w.block_size
            tiles.append((to_dev(blocks), to_dev(counts), to_dev(last)))
    ctx = pda.Context(max_seqs=w.B * args.q_len, num_q_heads=w.Hq, num_kv_heads=w.Hkv,
                      head_dim=w.D, block_size=w.block_size, tile_capacity=tile_cap)
    ctx.set_multi_tc(args.multi_form == "tc")
    stream = torch.cuda.current_stream()

    def call(s, out):
        """One decode of input set s into out through the public API."""
        if args.tiles > 0:
            ctx.begin_step(w.B)
            for blocks, counts, last in tiles:
                ctx.step_tile(s["q"], s["k_pool"], s["v_pool"], blocks, counts, last)
            ctx.finalize(w.B, out=out)
        elif args.q_len > 1:
            ctx.decode_multi(s["q"], s["k_pool"], s["v_pool"], s["block_table"], s["seq_lens"],
                             out=out)
        elif args.layout == "contiguous":
            ctx.decode_contiguous(s["q"], s["k_pool"], s["v_pool"], s["seq_lens"], out=out)
        else:
            ctx.decode(s["q"], s["k_pool"], s["v_pool"], s["block_table"], s["seq_lens"], out=out)

    counter = [0]

    def step(_k=None):
        # consecutive calls always read a different input set (L2 is never warm)
        i = counter[0]
        counter[0] += 1
        call(sets[i % n_sets], outs[i % n_sets])

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if ctx.read_device_errors() != 0:
        raise RuntimeError("device error flags set during warm-up")

    # --- main timed region: exactly K calls, back to back
    pad_s = 0.0 if args.quick else 0.6  # keep the GPU busy while the sampler starts
    sampler = ClockSampler(local_rank)
    if not args.quick:
        sampler.start()
    t_pad0 = time.time()
    pad_end = time.time() + pad_s
    i = 0
    while time.time() < pad_end:
        step(i); i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    graph = None
    if not args.no_graph:
        # the K calls, with their input-set rotation, captured once
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for k in range(args.steps):
                    step(k)
        stream.wait_stream(cap)
        graph.replay()  # warm
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(args.steps):
            step(k)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_total = e0.elapsed_time(e1)
    # the same calls launched one by one from Python (host launch cost included)
    a_l, b_l = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_l.record(stream)
    for k in range(args.steps):
        step(k)
    b_l.record(stream)
    torch.cuda.synchronize()
    loop_us = a_l.elapsed_time(b_l) * 1e3 / args.steps
    pad_end = time.time() + pad_s
    while time.time() < pad_end:
        step(i); i += 1
        if i % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    t_pad1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_pad0, t_pad1)
    clocks["window"] = "timed calls plus 0.6 s of the same calls on either side"

    ms_step = max_over_ranks(ms_total / args.steps, dev)

    # --- kernel timing pass: events around the split kernel of each call
    # (one-shot calls only; a tiled step is timed as a whole)
    n_timed = 0 if (args.quick or args.tiles > 0) else args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(n_timed)]
    for k in range(n_timed):
        # torch only computes elapsed times of events it recorded itself; the
        # library re-records the same events later, and the last record wins
        for e in evs[k]:
            e.record(stream)
        ctx.set_timing_events(*evs[k])
        step(k)
    ctx.set_timing_events(None, None, None)
    torch.cuda.synchronize()
    split_ms = [a.elapsed_time(b) for a, b, _ in evs]
    split_avg = statistics.mean(split_ms) if split_ms else float("nan")
    if ctx.read_device_errors() != 0:
        raise RuntimeError("device error flags set during timing")

    # --- per-call distribution: an event pair around each call (events between
    # calls stop the next call's early launch, so these are isolated calls)
    per_call = None
    if not args.quick:
        n_pc = max(50, min(args.steps, 200))
        pc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_pc)]
        for a, b in pc:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        us = sorted(a.elapsed_time(b) * 1e3 for a, b in pc)
        per_call = {"median": statistics.median(us), "p10": us[int(0.1 * (n_pc - 1))],
                    "p90": us[int(0.9 * (n_pc - 1))], "calls": n_pc,
                    "note": "isolated calls, inputs rotated (L2 cold)"}

    # --- L2-warm number (same inputs every call) for the workloads that fit in L2
    l2_warm = None
    if not args.quick and input_bytes < l2 // 2:
        s0, o0 = sets[0], outs[0]

        def warm_step():
            call(s0, o0)

        for _ in range(5):
            warm_step()
        torch.cuda.synchronize()
        warm_graph = None
        if not args.no_graph:
            warm_graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(warm_graph, stream=cap):
                    for _ in range(args.steps):
                        warm_step()
            stream.wait_stream(cap)
            warm_graph.replay()
            torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if warm_graph is not None:
            warm_graph.replay()
        else:
            for _ in range(args.steps):
                warm_step()
        b.record(stream)
        torch.cuda.synchronize()
        warm_us = a.elapsed_time(b) * 1e3 / args.steps
        l2_warm = {"us_per_call": warm_us, "GB/s": bytes_per_call / (warm_us * 1e-6) / 1e9,
                   "note": "L2-warm: one input set reused every call (labelled; not the metric)"}

    # --- end to end: pinned host inputs copied in, output copied back, each step
    e2e = None
    if not (args.no_e2e or args.quick):
        pinned = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).pin_memory()
                  for k, v in host.items()}
        out_host = torch.empty(tuple(outs[0].shape), dtype=torch.bfloat16).pin_memory()
        dst = sets[0]
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        d2h = out_host.numel() * out_host.element_size()
        k_e2e = max(3, min(args.steps, 50))

        def e2e_step():
            for k, t in pinned.items():
                d = dst[k].view(torch.int16) if dst[k].dtype == torch.bfloat16 else dst[k]
                d.copy_(t, non_blocking=True)
            call(dst, outs[0])
            out_host.copy_(outs[0], non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / k_e2e, dev)
        e2e = {"value": world * bytes_per_call / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "us_per_call": e2e_ms * 1e3, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": k_e2e}

    peak, peak_kind = peaks()
    value = world * bytes_per_call / (ms_step * 1e-3) / 1e9
    if args.tiles > 0 or args.quick:  # no split-kernel events
        split_avg = float("nan")
    # A decode call is one split-kernel launch, so the kernel's average launch
    # duration over the timed region (CUDA events around the K launches on their
    # stream) is the per-call time; a tiled step is its split launches plus the
    # reset and finalize kernels, reported as a whole.
    achieved = bytes_per_call / (ms_step * 1e-3) / 1e9
    info = ctx.launch_info()
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "us_per_call": ms_step * 1e3,
        "loop_us_per_call": loop_us,
        "pct_of_hbm_peak": 100.0 * value / (world * peak),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) q/K/V rounded to bf16, shuffled block table",
        "config": {**w.describe(), "workload": w.name, "kv_layout": args.layout,
                   "q_len": args.q_len, "tiles": args.tiles,
                   **({"multi_form": ["n8", "row form (mma.sync)", "row form (tcgen05)"][
                       ctx.multi_info(args.q_len)["form"]]} if args.q_len > 1 else {}),
                   "l2": f"inputs larger than L2 ({input_bytes / 1e6:.0f} MB per set, "
                         f"{n_sets} sets rotated, L2 {l2 / 2 ** 20:.0f} MiB)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": ("K calls replayed from one CUDA graph" if graph is not None
                              else "K calls launched one by one"),
                   "split_ctas": info["split_ctas"], "ctas_per_sm": info["ctas_per_sm"],
                   "stages": info["stages"], "algorithmic_bytes_per_call": bytes_per_call},
        "roofline": {"bound": "hbm",
                     "kernel": ("split_kernel (one launch per call)" if args.tiles == 0
                                else "tiled step (reset, one split launch per tile, finalize)"),
                     "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs (STREAM-style copy)", "unit": "GB/s",
                     "frac": achieved / peak,
                     # the ncu record holds the default configuration of each workload
                     "traffic": (recorded_traffic(args.workload)
                                 if (args.block_size == 0 and args.layout == "paged"
                                     and args.q_len == 1 and args.tiles == 0) else None),
                     "launch_us": ms_step * 1e3,
                     "timing": ("achieved = algorithmic bytes / the split kernel's average "
                                "launch duration over the timed region (CUDA events around the "
                                "K graph-replayed launches on their stream; one launch per "
                                "call; consecutive launches overlap their set-up, and the next "
                                "launch's prefetch warp moves its first stages into L2 while "
                                "the previous one finishes)"),
                     "isolated_us": None if math.isnan(split_avg) else split_avg * 1e3,
                     "isolated_timing": ("the kernel with CUDA events before and after every "
                                         "launch, which also stops the next launch's early "
                                         "set-up: the launch gap is included")},
        # one split kernel per call; a tiled step: reset, one split kernel per tile, finalize
        "gpu_launches": (2 + args.tiles if args.tiles > 0 else 1) * args.steps,
        "clocks": clocks,
    }
    if per_call is not None:
        line["per_call_us"] = per_call
    if l2_warm is not None:
        line["l2_warm"] = l2_warm
    if e2e is not None:
        line["e2e"] = e2e
    default_config = (args.workload == "8b" and args.block_size == 0 and args.q_len == 1
                      and args.tiles == 0 and args.layout == "paged")
    if rank == 0 and not (args.quick or args.no_others) and default_config:
        line["other_configs"] = {name: time_other_config(name, dev, max(10, min(args.steps, 50)),
                                                         args.warmup, peak)
                                 for name in OTHER_CONFIGS}
    if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.quick):
        cb = cpu_oracle_timing(w)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                   "single_thread")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
