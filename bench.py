#!/usr/bin/env python
"""Benchmark of batched heterogeneous sampling (+ speculative verification).

Headline: sampled rows/s and logits-read HBM GB/s on the heterogeneous-decode
workload (64 rows x V = 128256, bf16 logits, every row with penalties over a
512-id history, 16 bias entries, mixed greedy / top-k / top-p / min-p).

A step is one ss_process_sample call on one 64-row batch.  Steps cycle through
a ring of input sets whose total size exceeds twice the L2 cache, so every
step reads its logits from HBM.  The K timed steps are replayed from CUDA
graphs (a graph of `ring * 8` calls, replayed) and timed with CUDA events on
the launching stream, between barriers and device synchronisations; the
maximum over ranks is reported.  Multi-GPU runs are data-parallel replicas
(weak scaling: every rank samples its own batches; no collective on the data
path).

--impl reference times the CPU oracle (the plain single-threaded C program
under oracle/) on the same workload and metric, as the reference arm.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_verification_gb300 import dp as DP  # noqa: E402
from speculative_verification_gb300 import workloads as W  # noqa: E402

METRIC = "sampled rows/s and logits HBM GB/s (% of peak) at V=128k B=64; spec-verify rows/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
KERNEL_NAME = "ss_hist_kernel"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def progress(msg):
    """Phase markers on stderr (flushed), so that a stalled run shows where."""
    if os.environ.get("SS_BENCH_PROGRESS"):
        print("[bench %.1fs] %s" % (time.time() - _T0, msg), file=sys.stderr, flush=True)


_T0 = time.time()


KERNEL_SOURCES = {
    "ss_hist_kernel": ("ss_hist.cu", "ss_hist.h"),
    "ss_row_kernel": ("ss_kernel.cu",),
    "ss_fused_kernel": ("ss_fused.cu",),
}


def _code_only(text):
    """C / CUDA source without its comments and blank lines (the sources hold
    no comment markers inside string literals), so that editing a comment
    does not count as changing the kernel."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel=KERNEL_NAME):
    """Hash of the code one kernel is compiled from: its translation unit(s),
    the shared device headers and the C header, comments left out."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_verification_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + ("ss_philox.cuh", "ss_ptx.cuh"):
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    with open(os.path.join(ROOT, "include", "ss.h")) as f:
        h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload_key, kernel=KERNEL_NAME):
    """Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum)
    recorded from an ncu capture in profiles/traffic.json, if that capture
    was taken on the current source of the kernel and on this workload;
    otherwise None."""
    try:
        with open(TRAFFIC_FILE) as f:
            entries = json.load(f)["entries"]
    except (OSError, ValueError, KeyError):
        return None
    want = kernel_source_hash(kernel)
    for e in entries:
        if e.get("kernel") == kernel and e.get("kernel_sha256") == want and e.get("workload") == workload_key:
            try:
                return int(e["traffic_bytes_per_launch"])
            except (KeyError, ValueError, TypeError):
                return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.15)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_for(w):
    """The kernel a call on workload w runs: bf16 logits take the histogram
    kernel, fp32 logits the general row kernel."""
    return "ss_hist_kernel" if w["dtype"] == "bf16" else "ss_row_kernel"


def launches_per_call(w, cs):
    """Kernel launches one call makes: one for bf16 logits; the fp32 kernel
    gives the heavy rows (top-p without top-k) a concurrent launch of their
    own when there are 16 rows or more and the cluster can double."""
    if w["dtype"] == "bf16":
        return 1
    return 2 if (w["kind"] == "sample" and 16 <= int(w["num_rows"]) <= 4096 and 2 <= cs <= 4) else 1


def workload_for(cfg, rank, idx):
    return W.make(cfg, seed=DP.ring_seed(cfg, rank, idx))


# --------------------------------------------------------------- our arm --


def run_ours(args, rank, world, dist):
    import torch
    from speculative_verification_gb300 import build as ss_build
    from speculative_verification_gb300 import ss

    ss_build.build()
    ss.load()
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    cfg = args.config
    ring_host = [workload_for(cfg, rank, i) for i in range(args.ring)]
    bytes_per_call = W.algorithmic_bytes(ring_host[0])
    # kernel launches per sampling call: with 16 rows or more and a cluster
    # that can double, the heavy rows (top-p without top-k) get a concurrent
    # launch of their own with twice the CTAs per row
    cs = ss.ss_cluster_size(int(ring_host[0]["vocab"]), ring_host[0]["dtype"])
    per_call = launches_per_call(ring_host[0], cs)
    rows_per_call = int(ring_host[0]["num_rows"]) if ring_host[0]["kind"] == "sample" else int(
        ring_host[0]["draft_offsets"][-1]) + int(ring_host[0]["num_requests"])
    ring = [ss.to_device(w, dev) for w in ring_host]
    out = ss.alloc_outputs(ring[0], dev)
    stream = torch.cuda.Stream(device=dev)

    # consecutive calls over independent batches may overlap (a call's first
    # rows start on the SMs the previous call's last rows leave:
    # SS_SAMPLE_OVERLAP_PREVIOUS / SS_VERIFY_OVERLAP_PREVIOUS); no call reads
    # another's outputs here
    overlap = ring_host[0]["kind"] in ("sample", "verify") and not args.no_overlap

    def call(i, ov=overlap):
        ss.run(ring[i % args.ring], out, stream=stream, overlap_previous=ov, target_rows=True)

    # graphs: one of `per_graph` calls (replayed), one for the remainder
    per_graph = min(args.steps, args.ring * 8)
    with torch.cuda.stream(stream):
        for i in range(args.ring):  # warm the launch path before capture
            call(i)
    stream.synchronize()

    def capture(n, ov=overlap):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(i, ov)
        return g

    progress("capturing graphs")
    g_main = capture(per_graph) if per_graph > 0 else None
    reps, rem = divmod(args.steps, per_graph) if per_graph > 0 else (0, 0)
    g_rem = capture(rem) if rem else None

    def replay_steps(n_steps):
        r, m = divmod(n_steps, per_graph)
        with torch.cuda.stream(stream):
            for _ in range(r):
                g_main.replay()
            if m:
                (g_rem if m == rem else capture(m)).replay()

    # warm-up (untimed)
    progress("warm-up replay")
    replay_steps(max(args.warmup, 3))
    stream.synchronize()

    # timed region
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        marks = []  # an event after every replay: best and median per replay
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g_main.replay()
                marks.append(torch.cuda.Event(enable_timing=True))
                marks[-1].record(stream)
            if g_rem is not None:
                g_rem.replay()
        stop.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    ms = start.elapsed_time(stop)
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    per_call_s = ms / 1e3 / args.steps
    value = DP.aggregate_rate(rows_per_call, args.steps, world, ms)
    per_replay = [a.elapsed_time(b) * 1e3 / per_graph for a, b in zip([start] + marks[:-1], marks)]
    # single calls without a graph, synchronised one by one (launch latency included)
    single = []
    for i in range(50):
        a_ev = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        with torch.cuda.stream(stream):
            call(i)
        b_ev.record(stream)
        stream.synchronize()
        single.append(a_ev.elapsed_time(b_ev) * 1e3)
    # the same graph of calls without the overlap: each call alone on the GPU
    alone_us = None
    if overlap and per_graph > 0:
        g_alone = capture(per_graph, False)
        with torch.cuda.stream(stream):
            g_alone.replay()
        stream.synchronize()
        a_ev = torch.cuda.Event(enable_timing=True)
        b_ev = torch.cuda.Event(enable_timing=True)
        a_ev.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_alone.replay()
        b_ev.record(stream)
        stream.synchronize()
        alone_us = a_ev.elapsed_time(b_ev) * 1e3 / (3 * per_graph)
        del g_alone
    call_us = {"mean": ms * 1e3 / args.steps,
               "best_replay": min(per_replay) if per_replay else None,
               "median_replay": statistics.median(per_replay) if per_replay else None,
               "one_call_at_a_time_in_graph": alone_us if overlap else ms * 1e3 / args.steps,
               "single_call_no_graph_median": statistics.median(single)}

    progress("timed region done: %.3f ms" % ms)
    # untimed: the GPU's outputs on the first input set, checked against the
    # oracle (all rows)
    chk = ss.alloc_outputs(ring[0], dev)
    ss.run(ring[0], chk, stream=stream, target_rows=True)
    stream.synchronize()
    gpu0 = {k: v.cpu().numpy() for k, v in chk.items() if k not in ("workspace", "processed")}
    n_check = int(ring_host[0]["num_rows"]) if ring_host[0]["kind"] == "sample" else int(ring_host[0]["num_requests"])
    parity = cpu_leg_check(ring_host[0], gpu0, range(n_check))["parity"] if not args.no_cpu_baseline else None
    progress("parity check done")

    # end-to-end through the public API with host buffers (pinned)
    e2e = run_e2e(args, ss, ring_host, dev, stream, rows_per_call, dist)
    progress("end-to-end done")

    # speculative-verify throughput (secondary metric), same protocol
    spec = run_spec(args, ss, rank, dev, stream) if args.spec_steps > 0 else None
    progress("spec-verify done")
    tree = run_tree(args, ss, rank, dev, stream) if args.tree_steps > 0 else None
    progress("tree-verify done")
    sharded = run_sharded(args, ss, rank, dev, stream) if args.shard_steps > 0 else None
    progress("sharded done")
    fused = run_fused(args, ss, dev, stream, measured_peak()[0]) if args.fused_steps > 0 else None
    progress("fused done")
    peak, peak_kind = measured_peak()
    grammar = mixed = None
    if args.grammar_calls > 0:
        grammar = run_config_block(args, ss, 3, rank, dev, stream, peak, 8, args.grammar_calls,
                                   range(128) if not args.no_cpu_baseline else [])
        progress("grammar done")
    if args.mixed_calls > 0:
        mixed = run_config_block(args, ss, 5, rank, dev, stream, peak, 1, args.mixed_calls,
                                 range(0, 256, 4) if not args.no_cpu_baseline else [])
        progress("mixed stress done")

    achieved = bytes_per_call / per_call_s / 1e9
    res = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64: bf16 N(0,3) logits + 1-5 spikes, mixed per-row params)",
        "config": {
            "workload": W.CONFIG_NAMES[cfg],
            "rows_per_step": rows_per_call,
            "vocab": int(ring_host[0]["vocab"]),
            "input_dtype": ring_host[0]["dtype"],
            "l2": "ring of %d input sets, %.0f MB > 2x L2" % (args.ring, args.ring * bytes_per_call / 1e6),
            "launch": ("CUDA graph of %d calls, replayed; consecutive calls overlap (programmatic dependent "
                       "launch, %s)" % (per_graph, "SS_SAMPLE_OVERLAP_PREVIOUS" if ring_host[0]["kind"] == "sample"
                                        else "SS_VERIFY_OVERLAP_PREVIOUS")) if overlap else (
                           "CUDA graph of %d calls, replayed" % per_graph),
            "parallelism": "dp%d replicas" % world,
            "cluster_ctas_per_row": cs,
            "launches_per_call": per_call,
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "frac_of_nominal_7900": achieved / 7900.0,
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind if peak_kind == "measured" else "fallback",
            "algorithmic_bytes_per_launch": bytes_per_call,
            "traffic": recorded_traffic(W.CONFIG_NAMES[cfg], kernel_for(ring_host[0])),
            "kernel": kernel_for(ring_host[0]),
            "kernel_sha256": kernel_source_hash(kernel_for(ring_host[0])),
        },
        "e2e": e2e,
        "us_per_call": call_us,
        "gpu_launches": args.steps * per_call,
        "clocks": clocks.summary(),
    }
    if spec is not None:
        res["spec_verify"] = spec
    if tree is not None:
        res["tree_verify"] = tree
    if sharded is not None:
        res["vocab_sharded"] = sharded
    if fused is not None:
        res["fused_lmhead"] = fused
    if parity is not None:
        res["parity"] = parity
    if grammar is not None:
        res["grammar"] = grammar
    if mixed is not None:
        res["mixed_stress"] = mixed
    return res


def run_e2e(args, ss, ring_host, dev, stream, rows_per_call, dist):
    """Same metric through ss_process_sample with the step's inputs copied from
    pinned host memory and the results copied back, every step.  Each input
    set is one pinned buffer (one copy per step); two device staging buffers
    let step i+1's copy run on a copy stream while step i samples, as a
    serving loop would overlap them."""
    import torch
    n_steps = max(2, min(args.e2e_steps, args.steps))
    sets = ring_host[: min(4, len(ring_host))]
    lay, total = ss.pack_layout(sets[0])
    pinned = [ss.pack_pinned(w, lay, total) for w in sets]
    bufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    staging = [ss.views(b, lay, sets[0]) for b in bufs]
    # output sizes from the host copy: the staging buffers are not filled yet
    outs = [ss.alloc_outputs(sets[0], dev) for _ in staging]
    keys = [k for k in ("token", "status", "kept", "out_tokens", "num_accepted") if k in outs[0]]
    host_out = [{k: torch.empty(o[k].shape, dtype=o[k].dtype, pin_memory=True) for k in keys} for o in outs]
    h2d = sum(lay[k][1] for k in lay)
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())
    copy_stream = torch.cuda.Stream(device=dev)  # host to device, back to back
    back_stream = torch.cuda.Stream(device=dev)  # device to host (the link's other direction)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]

    def h2d_copy(i):
        b = i % 2
        if i >= 2:
            copy_stream.wait_event(done[b])  # step i-2 has finished reading this staging buffer
        with torch.cuda.stream(copy_stream):
            bufs[b].copy_(pinned[i % len(pinned)], non_blocking=True)
            copied[b].record(copy_stream)

    def sample(i):
        b = i % 2
        stream.wait_event(copied[b])
        if i >= 2:
            stream.wait_event(read[b])  # step i-2's results are read back from these outputs
        with torch.cuda.stream(stream):
            ss.run(staging[b], outs[b], stream=stream)
            done[b].record(stream)

    def d2h_copy(i):
        b = i % 2
        back_stream.wait_event(done[b])
        with torch.cuda.stream(back_stream):
            for k in keys:
                host_out[b][k].copy_(outs[b][k], non_blocking=True)
            read[b].record(back_stream)

    def steps(n):
        # the input copies run back to back on one stream (the host link is
        # the bound), step i samples once its copy has landed, and its results
        # go back on a third stream; a staging buffer is refilled once the
        # step two before has sampled from it, and its outputs rewritten once
        # they are read back
        for i in range(n):
            h2d_copy(i)
            if i >= 1:
                sample(i - 1)
                d2h_copy(i - 1)
        sample(n - 1)
        d2h_copy(n - 1)

    steps(4)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(copy_stream)
    steps(n_steps)
    t1.record(back_stream)  # after the last read-back, which follows every copy and call
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    # the last step's read-back equals a plain call on the same input set
    last = n_steps - 1
    ref_in = ss.to_device(sets[last % len(sets)], dev)
    ref_out = ss.alloc_outputs(ref_in, dev)
    ss.run(ref_in, ref_out)
    torch.cuda.synchronize()
    for k in keys:
        if not torch.equal(host_out[last % 2][k], ref_out[k].cpu()):
            raise RuntimeError("pipelined end-to-end results differ from a direct call (%s)" % k)
    if dist:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    world = dist.get_world_size() if dist else 1
    return {"value": DP.aggregate_rate(rows_per_call, n_steps, world, ms), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n_steps,
            "pipeline": "one packed copy per step, back to back on a copy stream, overlapped with the previous step's sampling; read-backs on a third stream"}


def graph_of_calls(ss, ring, out, stream, overlap, min_calls=16):
    """A CUDA graph of consecutive calls cycling through the input sets of
    `ring` (whole passes, at least `min_calls` calls), so that consecutive
    calls may overlap inside it as in a serving loop; verification calls
    state their number of target rows.  Returns the graph and its number of
    calls."""
    import torch
    inner = max(1, -(-min_calls // len(ring)))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(inner):
                for dw in ring:
                    ss.run(dw, out, stream=stream, overlap_previous=overlap, target_rows=True)
    return g, inner * len(ring)


def run_spec(args, ss, rank, dev, stream):
    """Verification throughput on the linear-draft workload (32 requests, k=4)."""
    import torch
    ring_host = [workload_for(4, rank, i) for i in range(max(2, args.ring // 2))]
    ring = [ss.to_device(w, dev) for w in ring_host]
    out = ss.alloc_outputs(ring[0], dev)
    rows = int(ring_host[0]["draft_offsets"][-1]) + int(ring_host[0]["num_requests"])
    with torch.cuda.stream(stream):
        ss.ss_workspace_init(out["workspace"], stream=stream)
        for i in range(len(ring)):
            ss.run(ring[i], out, stream=stream, overlap_previous=not args.no_overlap, target_rows=True)
    stream.synchronize()
    g, per_graph = graph_of_calls(ss, ring, out, stream, not args.no_overlap)
    reps = max(1, args.spec_steps // per_graph)
    with torch.cuda.stream(stream):  # warm-up on the timed stream, finished before t0
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    calls = reps * per_graph
    # the step after verification (tokens placed for the next step on the
    # device), timed on its own
    R, width = out["out_tokens"].shape
    cap = 4096
    tokens = torch.zeros((R, cap), dtype=torch.int32, device=dev)
    seq = torch.zeros(R, dtype=torch.int32, device=dev)
    pos = torch.zeros(R, dtype=torch.int64, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)
    cst = torch.empty(R, dtype=torch.int32, device=dev)
    gc = torch.cuda.CUDAGraph()
    n_commit = 256
    with torch.cuda.stream(stream):
        with torch.cuda.graph(gc, stream=stream):
            for _ in range(n_commit):
                ss.ss_commit_accepted(out["out_tokens"], out["num_accepted"], out["status"], tokens, seq, pos, nxt,
                                      cst, stream=stream)
    with torch.cuda.stream(stream):
        seq.zero_()
        gc.replay()
        seq.zero_()
    stream.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    with torch.cuda.stream(stream):
        gc.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    commit_us = c0.elapsed_time(c1) * 1e3 / n_commit
    return {"workload": W.CONFIG_NAMES[4], "target_rows_per_s": rows * calls / (ms / 1e3),
            "commit_accepted_us_per_call": commit_us,
            "requests_per_s": int(ring_host[0]["num_requests"]) * calls / (ms / 1e3),
            "ms_per_call": ms / calls, "calls": calls,
            "logits_GBps": W.algorithmic_bytes(ring_host[0]) * calls / (ms / 1e3) / 1e9,
            "consecutive_calls_overlap": not args.no_overlap, "calls_per_graph": per_graph,
            "target_rows_stated": True}


TREE_WORKLOAD = "tree verify R=32 trees of 1-16 nodes V=128256 bf16"


def run_tree(args, ss, rank, dev, stream):
    """Tree-draft verification: 32 requests, random draft trees of 1 to 16
    nodes (each node under one of the 4 nodes before it), V = 128256 bf16,
    drafts drawn from a noisy copy of each node's target row."""
    import torch
    ring_host = [W.tree(seed=9000 + 97 * rank + i, requests=32, vocab=128256, max_nodes=16) for i in range(3)]
    ring = [ss.to_device(w, dev) for w in ring_host]
    out = ss.alloc_outputs(ring[0], dev)
    rows = sum(int(w["node_offsets"][-1]) for w in ring_host)
    with torch.cuda.stream(stream):
        ss.ss_workspace_init(out["workspace"], stream=stream)
        for dw in ring:
            ss.run(dw, out, stream=stream, overlap_previous=not args.no_overlap)
    stream.synchronize()
    g, per_graph = graph_of_calls(ss, ring, out, stream, not args.no_overlap)
    reps = max(1, args.tree_steps // per_graph)
    with torch.cuda.stream(stream):  # warm-up on the timed stream, finished before t0
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    calls = reps * per_graph
    passes = calls // len(ring)  # whole passes over the ring
    alg = sum(W.algorithmic_bytes(w) for w in ring_host)
    return {"workload": TREE_WORKLOAD, "node_rows_per_s": rows * passes / (ms / 1e3),
            "requests_per_s": 32 * calls / (ms / 1e3), "ms_per_call": ms / calls, "calls": calls,
            "mean_nodes_per_request": rows / (32.0 * len(ring)),
            "logits_GBps": alg * passes / (ms / 1e3) / 1e9, "consecutive_calls_overlap": not args.no_overlap,
            "calls_per_graph": per_graph, "target_rows_stated": True}


def run_sharded(args, ss, rank, dev, stream, parts=4):
    """The vocabulary-sharded path on one GPU, on the headline workload as it
    is: `parts` shard launches and one merge for the top-k rows (the list
    path), then four rounds of `parts` shard launches and one merge for the
    top-p / min-p rows without top-k, all into the same outputs.  The shards
    of a step run on one stream each (on P GPUs they would run at the same
    time), forked from and joined back into the call's stream."""
    import torch
    ring_host = [workload_for(2, rank, i) for i in range(max(2, args.ring // 2))]
    ring = [ss.to_device(w, dev) for w in ring_host]
    n = int(ring_host[0]["num_rows"])
    V = int(ring_host[0]["vocab"])
    cap = 1024
    bounds = W.even_shards(V, parts)
    recs = [torch.empty(n * ss.ss_shard_record_bytes(cap), dtype=torch.uint8, device=dev) for _ in bounds]
    rrecs = [torch.empty(n * ss.ss_shard_round_record_bytes(), dtype=torch.uint8, device=dev) for _ in bounds]
    state = torch.empty(ss.ss_shard_round_state_bytes(n), dtype=torch.uint8, device=dev)
    tok = torch.empty(n, dtype=torch.int32, device=dev)
    st = torch.empty(n, dtype=torch.int32, device=dev)
    kept = torch.empty(n, dtype=torch.int32, device=dev)
    shard_streams = [torch.cuda.Stream(device=dev) for _ in bounds]
    fork = torch.cuda.Event()
    joins = [torch.cuda.Event() for _ in bounds]

    def shards(launch):
        fork.record(stream)
        for i, (sst, jn) in enumerate(zip(shard_streams, joins)):
            sst.wait_event(fork)
            launch(i, sst)
            jn.record(sst)
        for jn in joins:
            stream.wait_event(jn)

    def call(dw):
        params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
        params["bitmask_stride"] = dw.get("bitmask_stride", 0)
        stride = int(dw["row_stride"])

        def list_shard(i, sst):
            off, length = bounds[i]
            ss.ss_sample_shard(dw["logits"][:, off:], params, recs[i], vocab=V, vocab_offset=off, shard_len=length,
                               list_cap=cap, num_rows=n, dtype=dw["dtype"], row_stride=stride, stream=sst)
        shards(list_shard)
        ss.ss_merge_shards(recs, params, tok, st, vocab=V, list_cap=cap, out_kept=kept, stream=stream)
        for rnd in range(4):
            def round_shard(i, sst, rnd=rnd):
                off, length = bounds[i]
                ss.ss_shard_round(dw["logits"][:, off:], params, state, rrecs[i], round=rnd, vocab=V,
                                  vocab_offset=off, shard_len=length, num_rows=n, dtype=dw["dtype"],
                                  row_stride=stride, stream=sst)
            shards(round_shard)
            ss.ss_merge_round(rrecs, params, state, tok, st, round=rnd, vocab=V, out_kept=kept, stream=stream)

    with torch.cuda.stream(stream):
        for dw in ring:
            call(dw)
    stream.synchronize()
    # the sharded outputs of the last input set equal a single call's
    ref = ss.alloc_outputs(ring[-1], dev)
    ss.run(ring[-1], ref, stream=stream)
    stream.synchronize()
    same = all(torch.equal(x, ref[k]) for x, k in ((tok, "token"), (st, "status"), (kept, "kept")))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for dw in ring:
                call(dw)
    reps = max(1, args.shard_steps // len(ring))
    with torch.cuda.stream(stream):  # warm-up on the timed stream, finished before t0
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    calls = reps * len(ring)
    return {"workload": W.CONFIG_NAMES[2], "shards": len(bounds),
            "rows_per_s": n * calls / (ms / 1e3), "ms_per_call": ms / calls, "calls": calls,
            "launches_per_call": 5 * (len(bounds) + 1),
            "equal_to_single_call": bool(same),
            "path": "top-k rows: one shard launch each + merge; top-p / min-p rows without top-k: four rounds "
                    "of one launch per shard + merge; shard launches concurrent, one stream each"}


def run_fused(args, ss, dev, stream, peak):
    """The LM head fused with the draw (B=64, d=4096, V=128256 bf16): the
    weight matrix (1.05 GB, larger than L2) is streamed from HBM every call;
    roofline = weight + hidden-state bytes per call over the call's time."""
    import torch
    B, d, V = 64, 4096, 128256
    gen = torch.Generator(device=dev)
    gen.manual_seed(6)
    h = torch.randn(B, d, device=dev, generator=gen).to(torch.bfloat16)
    wt = (torch.randn(V, d, device=dev, generator=gen) * (3.0 / d ** 0.5)).to(torch.bfloat16)
    temp = torch.rand(B, device=dev, generator=gen) + 0.5
    seed = torch.arange(B, device=dev, dtype=torch.int64) + 1000
    pos = torch.zeros(B, device=dev, dtype=torch.int64)
    scratch = torch.empty(ss.ss_fused_scratch_bytes(B), dtype=torch.uint8, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)

    def call():
        ss.ss_fused_lmhead_sample(h, wt, temp, seed, pos, scratch, tok, st, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
    stream.synchronize()
    per_graph = 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(per_graph):
                call()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    reps = max(1, args.fused_steps // per_graph)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    calls = reps * per_graph
    ms = t0.elapsed_time(t1) / calls
    alg = V * d * 2 + B * d * 2
    ach = alg / (ms / 1e3) / 1e9
    return {"workload": "fused LM head + draw B=%d d=%d V=%d bf16" % (B, d, V), "kernel": "ss_fused_kernel",
            "rows_per_s": B / (ms / 1e3), "us_per_call": ms * 1e3, "calls": calls,
            "tflops": 2.0 * B * d * V / (ms / 1e3) / 1e12, "launches_per_call": 3,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                         "algorithmic_bytes_per_launch": alg,
                         "traffic": recorded_traffic("fused LM head + draw B=%d d=%d V=%d bf16" % (B, d, V),
                                                     "ss_fused_kernel"),
                         "kernel_sha256": kernel_source_hash("ss_fused_kernel")}}


def run_config_block(args, ss, cfg, rank, dev, stream, peak, ring_n, calls_wanted, check_reqs):
    """Throughput of one more workload (3: grammar-constrained, 5: mixed
    stress), timed like the headline: a ring of input sets larger than twice
    the L2 cache (or one set larger than it), calls replayed from a CUDA graph,
    CUDA events on the launching stream.  Afterwards (untimed) the GPU's
    outputs on the first set are checked against the oracle on `check_reqs`."""
    import torch
    progress("config %d: generating %d input sets" % (cfg, ring_n))
    ring_host = [workload_for(cfg, rank, i) for i in range(ring_n)]
    ring = [ss.to_device(w, dev) for w in ring_host]
    out = ss.alloc_outputs(ring[0], dev)
    w0 = ring_host[0]
    rows = int(w0["num_rows"]) if w0["kind"] == "sample" else int(w0["draft_offsets"][-1]) + int(w0["num_requests"])
    alg = W.algorithmic_bytes(w0)
    cs = ss.ss_cluster_size(int(w0["vocab"]), w0["dtype"])
    overlap = w0["kind"] in ("sample", "verify") and not args.no_overlap  # as the headline
    with torch.cuda.stream(stream):
        if "workspace" in out:
            ss.ss_workspace_init(out["workspace"], stream=stream)
        for dw in ring:
            ss.run(dw, out, stream=stream, overlap_previous=overlap, target_rows=True)
    stream.synchronize()
    g, per_graph = graph_of_calls(ss, ring, out, stream, overlap, min_calls=min(16, calls_wanted))
    reps = max(1, calls_wanted // per_graph)
    with torch.cuda.stream(stream):  # warm-up on the timed stream, finished before t0
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    calls = reps * per_graph
    per_call_s = ms / 1e3 / calls
    achieved = alg / per_call_s / 1e9
    # untimed: one more call on the first set, for the check
    chk = ss.alloc_outputs(ring[0], dev)
    ss.run(ring[0], chk, stream=stream, target_rows=True)
    stream.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in chk.items() if k not in ("workspace", "processed")}
    kernel = kernel_for(w0)
    block = {
        "workload": W.CONFIG_NAMES[cfg],
        "rows_per_call": rows,
        "rows_per_s": rows / per_call_s,
        "us_per_call": per_call_s * 1e6,
        "calls": calls,
        "gpu_launches": calls * launches_per_call(w0, cs),
        "l2": "ring of %d input set(s), %.0f MB%s" % (ring_n, ring_n * alg / 1e6,
                                                       " > 2x L2" if ring_n * alg > 2 * L2_BYTES else " > L2"),
        "consecutive_calls_overlap": overlap,
        "calls_per_graph": per_graph,
        "target_rows_stated": w0["kind"] == "verify",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes_per_launch": alg, "traffic": recorded_traffic(W.CONFIG_NAMES[cfg], kernel),
                     "kernel": kernel, "kernel_sha256": kernel_source_hash(kernel)},
    }
    if len(check_reqs):
        block.update(cpu_leg_check(w0, gpu, check_reqs))
    return block


# -------------------------------------------------------- oracle timing --


def cpu_leg_check(w, gpu, reqs):
    """The CPU-baseline leg on a checked sample: the oracle run on the
    requests `reqs` of input set w (timed: its rows/s on one thread), and the
    GPU's outputs for them compared with it as the parity tests do -- tokens,
    statuses and accepted counts must match except where the oracle marks the
    decision as within the 1e-5 margin; a GPU kept-set size inside the
    oracle's margin range is adopted (forced_kept counts those).  Reports
    counts; never raises on a mismatch."""
    from oracle import oracle as O
    reqs = list(reqs)
    sub = W.subset_requests(w, reqs)
    if w["kind"] == "sample":
        g = {k: gpu[k][reqs] for k in ("token", "status", "kept")}
        t0 = time.perf_counter()
        ref = O.process_sample(sub, force_kept=g["kept"])
        el = time.perf_counter() - t0
        ok = ref["status"] == 0
        forced = ok & (g["kept"] != ref["kept_own"])
        outside = ok & ((g["kept"] < ref["kept_lo"]) | (g["kept"] > ref["kept_hi"]))
        sm = ok & (ref["sub_margin"] != 0)
        mism = (g["status"] != ref["status"]) | (ok & ~sm & (g["token"] != ref["token"])) | outside
        rows = len(reqs)
    else:
        d = w["draft_offsets"]
        trows = np.concatenate([np.arange(int(d[r]) + r, int(d[r + 1]) + r + 1) for r in reqs])
        g = {"out_tokens": gpu["out_tokens"][reqs], "num_accepted": gpu["num_accepted"][reqs],
             "status": gpu["status"][reqs], "kept": gpu["kept"][trows]}
        t0 = time.perf_counter()
        ref = O.spec_verify(sub, force_kept=g["kept"])
        el = time.perf_counter() - t0
        ok = ref["status"] == 0
        off = sub["draft_offsets"]
        forced = np.zeros(len(reqs), bool)
        outside = np.zeros(len(reqs), bool)
        for i in range(len(reqs)):
            rr = np.arange(int(off[i]) + i, int(off[i + 1]) + i + 1)
            forced[i] = ok[i] and np.any(g["kept"][rr] != ref["kept_own"][rr])
            outside[i] = ok[i] and np.any((g["kept"][rr] < ref["kept_lo"][rr]) | (g["kept"][rr] > ref["kept_hi"][rr]))
        sm = ok & (ref["sub_margin"] != 0)
        tok_bad = np.array([not np.array_equal(g["out_tokens"][i], ref["out_tokens"][i]) for i in range(len(reqs))])
        mism = (g["status"] != ref["status"]) | (ok & ~sm & ((g["num_accepted"] != ref["num_accepted"]) | tok_bad)) | outside
        rows = int(len(trows))
    return {"parity": {"checked": len(reqs), "unit": "rows" if w["kind"] == "sample" else "requests",
                       "status_ok": int(ok.sum()), "mismatches": int(mism.sum()), "sub_margin": int(sm.sum()),
                       "forced_kept": int(forced.sum()),
                       "what": "GPU outputs of one input set against the CPU oracle, outside the timed region"},
            "cpu_oracle": {"value": rows / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
                           "sample": "%d target rows of the checked sample, one thread" % rows}}





def time_oracle(cfg, seconds, max_steps=None):
    """Rows/s of the CPU oracle on rows of the same workload (1 thread)."""
    from oracle import oracle as O
    sample = W.make(cfg, seed=cfg + 424242, rows=8) if cfg != 4 else None
    if sample is None:
        raise ValueError("oracle timing uses sampling workloads")
    rows = 0
    steps = 0
    t0 = time.perf_counter()
    while True:
        O.process_sample(sample)
        rows += int(sample["num_rows"])
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_steps and steps >= max_steps):
            break
    return rows / el, rows, el


def cpu_baseline_block(cfg, seconds):
    v, rows, el = time_oracle(cfg, seconds)
    return {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": "%d rows of the %s workload (8-row batches) in %.1f s, one thread" % (rows, W.CONFIG_NAMES[cfg], el)}


def cpu_parallel_block(cfg, seconds):
    """The same oracle on every host core at once: one thread per core, each
    sampling its own 8-row batches (rows are independent; the C oracle runs
    without the interpreter lock)."""
    import threading
    from oracle import oracle as O
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    samples = [W.make(cfg, seed=cfg + 424242 + i, rows=8) for i in range(cores)]
    O.process_sample(samples[0])  # build / load the oracle before the clock starts
    counts = [0] * cores
    t0 = time.perf_counter()

    def work(i):
        while time.perf_counter() - t0 < seconds:
            O.process_sample(samples[i])
            counts[i] += int(samples[i]["num_rows"])

    threads = [threading.Thread(target=work, args=(i,)) for i in range(cores)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    el = time.perf_counter() - t0
    rows = sum(counts)
    return {"value": rows / el, "unit": "rows/s", "cores": cores, "kind": "oracle, row-parallel",
            "sample": "%d rows of the %s workload (8-row batches) in %.1f s, %d threads" % (
                rows, W.CONFIG_NAMES[cfg], el, cores)}


def run_reference(args):
    """The oracle as the reference arm: each step samples one 8-row batch of
    the same workload; at most as many steps as fit in ~90 s are timed."""
    from oracle import oracle as O
    cfg = args.config
    sample = W.make(cfg, seed=cfg + 424242, rows=8)
    for _ in range(max(0, min(args.warmup, 2))):
        O.process_sample(sample)
    t0 = time.perf_counter()
    steps = 0
    budget = 90.0
    while steps < args.steps:
        O.process_sample(sample)
        steps += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    rows = steps * int(sample["num_rows"])
    value = rows / el
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": 1,
        "steps": steps,
        "steps_requested": args.steps,
        "warmup": args.warmup,
        "ms_per_step": el * 1e3 / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": W.CONFIG_NAMES[cfg], "rows_per_step": int(sample["num_rows"]),
                   "vocab": int(sample["vocab"])},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": "%d steps x 8 rows of the %s workload, one thread" % (steps, W.CONFIG_NAMES[cfg])},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, help="workload of the headline line: 2 (default), 1, 3 or 5")
    ap.add_argument("--ring", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--spec-steps", type=int, default=4000)
    ap.add_argument("--tree-steps", type=int, default=1500)
    ap.add_argument("--shard-steps", type=int, default=2000)
    ap.add_argument("--fused-steps", type=int, default=400)
    ap.add_argument("--grammar-calls", type=int, default=400, help="calls timed on workload 3 (0: skip)")
    ap.add_argument("--mixed-calls", type=int, default=20, help="calls timed on workload 5 (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="time calls one at a time (no SS_SAMPLE/VERIFY_OVERLAP_PREVIOUS)")
    args = ap.parse_args()

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by torchrun: start one process per GPU here, with the
        # same rendezvous variables torchrun would set
        return DP.launch_local(args.gpus, [sys.executable, os.path.abspath(__file__)] + sys.argv[1:])

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0

    # the oracle runs before any CUDA work (no fork after the first GPU call)
    cpu = cpu_par = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        progress("cpu baseline")
        cpu = cpu_baseline_block(args.config, args.cpu_seconds)
        cpu_par = cpu_parallel_block(args.config, max(2.0, args.cpu_seconds / 2))
        progress("cpu baseline done")

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if cpu is not None:
        res["cpu_baseline"] = cpu
        res["cpu_baseline_all_cores"] = cpu_par
    if rank == 0:
        print(json.dumps(res))
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
