#!/usr/bin/env python
"""Benchmark of the QSA selection step on GB300: query*blocks per second.

One step = one pass of the hot path over one query batch: the f32 queries
are converted to fp16, every block is scored (tensor-core full blocks, the
fp32 tail block with the +1e9 bonus) and the top-k blocks are selected per
query. Inputs are synthetic (qsa_inputs), resident in HBM, and the step
rotates through enough distinct input/output sets (> 2 x the 129 MB L2) that
every step reads its operands from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, on the host cores

Under torchrun every rank runs its own batches on its own GPU (no collective
on the data path); rank 0 prints one JSON line.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import qsa_inputs as qi  # noqa: E402

METRIC = "QSA score+top-k query·blocks/sec at 128K ctx, nq=256; % of GB300 roofline"
UNIT = "query*blocks/s"
DEFAULT_WORKLOAD = "long128k_nq256_h8_d128_kv131072"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by kernel, with the SHA-256 (first 16 hex
# digits) of the kernel's source files at capture time, or after a later edit
# that leaves the kernel's device code as captured (comments; host-side
# declarations in a shared header); an entry whose sources have changed
# otherwise reports null. The captures and their commands are summarised in
# profiles/.
NCU_TRAFFIC = {
    "fused_step_kernel": {"bytes_per_launch": 1651200,
                          "sources": ["fused_kernel.cuh", "select_row.cuh", "qsa_device.cuh"],
                          "source_sha": "0f670db82810e77e",
                          "workload": "long128k_nq256_h8_d128_kv131072"},
    "split_cluster_kernel": {"bytes_per_launch": 17340544,
                             "sources": ["split_reduce.cu", "qsa_device.cuh", "qsa_internal.h"],
                             "source_sha": "d789cc2cc8faa7dc",
                             "workload": "split_g4_r8_c128_b2048"},
}


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(qi.BY_NAME))
    p.add_argument("--batch", type=int, default=8,
                   help="query batches per launch for the batched measurement")
    p.add_argument("--min-timed-seconds", type=float, default=1.0,
                   help="repeat the K-step timed region until this much time has passed")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle baseline budget")
    p.add_argument("--no-split", action="store_true",
                   help="skip the split-reduce (second workload) measurement")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per-workload measurements (per_config)")
    p.add_argument("--per-config-cpu-seconds", type=float, default=1.5,
                   help="CPU oracle budget per workload in per_config")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "nq": w.nq, "H": w.H, "D": w.D, "n_kv": w.n_kv, "block": w.block,
           "nb": w.nb, "k": w.k, "q_input": "f32, converted to fp16 on the device in the step",
           "kb": "fp16, resident"}
    if extra:
        cfg.update(extra)
    return cfg


def units_per_step(w):
    return w.nq * w.nb


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="qsa_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax = [], []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                pass
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# -------------------------------------------------------------- GPU helpers
def rank_variants(rank, n):
    """The input-set variants rank `rank` draws: every rank processes its own
    independent query batches (weak scaling, no collective on the data)."""
    return range(rank * n, rank * n + n)


def max_over_ranks(torch, dist, value, device):
    """The largest of `value` over all ranks (the timing rule); `value` itself
    when there is one rank."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world, units_per_rank, ms):
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time."""
    return world * units_per_rank / (ms / 1e3)


class Sets:
    """Rotating device buffer sets for one workload, stored as contiguous
    [n, ...] tensors so that a slice of consecutive sets is itself a batch."""

    @staticmethod
    def bytes_per_set(w):
        return w.nq * w.H * w.D * (4 + 2) + w.nb * w.D * 2 + w.nq * w.nb * 4 + w.nq * w.k * 4

    def __init__(self, torch, tbs, w, device, min_bytes, rank=0, max_distinct=None, min_sets=2):
        per = Sets.bytes_per_set(w)
        n = max(min_sets, math.ceil(min_bytes / per))
        self.n = ((n + 7) // 8) * 8 if n > 8 else n  # whole groups of 8 for the batched launch
        self.per_set_bytes = per
        self.variants = rank_variants(rank, self.n)
        self.q32 = torch.empty((self.n, w.nq, w.H, w.D), dtype=torch.float32, device=device)
        self.kb = torch.empty((self.n, w.nb, w.D), dtype=torch.float16, device=device)
        # Small workloads need thousands of sets to exceed L2: draw up to
        # max_distinct seeded sets and fill the rest with copies of them (the
        # copies are distinct buffers, so every step still reads from HBM).
        distinct = self.n if max_distinct is None else min(self.n, max_distinct)
        for v, var in enumerate(list(self.variants)[:distinct]):
            q32, _ = qi.make_f32_inputs(w, variant=var)
            _, kb = qi.make_inputs(w, variant=var)
            self.q32[v].copy_(torch.from_numpy(q32))
            self.kb[v].copy_(torch.from_numpy(kb))
        for v0 in range(distinct, self.n, distinct):
            m = min(distinct, self.n - v0)
            self.q32[v0:v0 + m].copy_(self.q32[:m])
            self.kb[v0:v0 + m].copy_(self.kb[:m])
        self.q16 = torch.empty((self.n, w.nq, w.H, w.D), dtype=torch.float16, device=device)
        self.scores = torch.empty((self.n, w.nq, w.nb), dtype=torch.float32, device=device)
        self.ids = torch.empty((self.n, w.nq, w.k), dtype=torch.int32, device=device)
        # every q16 holds a converted copy so the score-only and select-only
        # timings read real data
        tbs.qsa_f32_to_f16(self.q32, out=self.q16)
        torch.cuda.synchronize()


def graph_of(torch, stream, fn, count):
    """Capture `count` calls fn(i) into one CUDA graph on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                fn(i)
    return g


def rotating_replay(torch, stream, fn, count, n_sets):
    """Graphs of exactly `count` calls each, graph j calling fn(j * count + i)
    for i < count, enough of them that together they touch all n_sets input
    sets; the returned replay() runs the next graph in turn. With n_sets
    sets larger than twice L2 in total, a set is touched again only after
    every other set has been, so each replay reads its inputs from HBM
    whatever `count` is."""
    n_graphs = max(1, -(-n_sets // count))
    graphs = [graph_of(torch, stream, lambda i, j=j: fn(j * count + i), count)
              for j in range(n_graphs)]
    state = {"next": 0}

    def replay():
        g = graphs[state["next"]]
        state["next"] = (state["next"] + 1) % n_graphs
        with torch.cuda.stream(stream):
            g.replay()
    for _ in range(n_graphs):  # upload + one untimed replay of each graph
        replay()
    return replay


def time_region(torch, stream, replay, reps_min, seconds, barrier=None, pre=None):
    """Time replay() (exactly K steps) with CUDA events on `stream`, repeated
    until `seconds` have passed (at least reps_min times). pre(), when given,
    runs before each timed region, outside it (the L2 flush). Returns the
    list of elapsed milliseconds, each the max over ranks."""
    out = []
    t_end = time.perf_counter() + seconds
    while len(out) < reps_min or time.perf_counter() < t_end:
        if barrier:
            barrier()
        if pre:
            pre()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        if barrier:
            ms = barrier(ms)
        out.append(ms)
        if len(out) >= 200:
            break
    return out


def kernel_source_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "top_block_selection_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel, w):
    e = NCU_TRAFFIC.get(kernel)
    if not e or e.get("workload") != w.name or e.get("source_sha") != kernel_source_sha(e["sources"]):
        return None
    return e["bytes_per_launch"]


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import top_block_selection_gb300 as tbs
    from top_block_selection_gb300 import _build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier(ms=None):
        if dist is None:
            return ms
        if ms is None:
            dist.barrier()
            return None
        return max_over_ranks(torch, dist, ms, device)

    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    _build.build()
    tbs.load_library()
    w = qi.BY_NAME[args.workload]
    K, W = args.steps, args.warmup
    if K < 1 or W < 3:
        raise SystemExit("need --steps >= 1 and --warmup >= 3")
    sets = Sets(torch, tbs, w, device, 2 * L2_BYTES, rank)
    stream = torch.cuda.Stream(device)
    peaks, peak_src = load_peaks()

    # Pass the fp16 query buffer only where it changes the library's plan
    # (large problems run the separate kernels, which need it); elsewhere the
    # fused launch would only write an extra copy of the queries.
    step_launches = tbs.qsa_select_step_launches(w.nq, w.H, w.D, w.n_kv, w.k, w.block, with_q16=False)
    with_q16 = tbs.qsa_select_step_launches(w.nq, w.H, w.D, w.n_kv, w.k, w.block,
                                            with_q16=True) != step_launches
    if with_q16:
        step_launches = tbs.qsa_select_step_launches(w.nq, w.H, w.D, w.n_kv, w.k, w.block,
                                                     with_q16=True)

    def step(i):
        v = i % sets.n
        tbs.qsa_select_step(sets.q32[v], sets.kb[v], w.n_kv, w.k, w.block,
                            q16=sets.q16[v] if with_q16 else None,
                            scores=sets.scores[v], ids=sets.ids[v])

    BB = args.batch

    n_launch = (K + BB - 1) // BB

    def batched(i):  # up to BB consecutive sets (one batch each) in one launch
        j, r = divmod(i, n_launch)   # graph j of the rotation, launch r in it
        nbat = min(BB, K - r * BB)
        v = (j * K + r * BB) % sets.n
        if v + nbat > sets.n:
            v = 0
        tbs.qsa_select_step_batched(sets.q32[v:v + nbat], sets.kb[v:v + nbat], w.n_kv, w.k,
                                    w.block, q16=sets.q16[v:v + nbat], scores=sets.scores[v:v + nbat],
                                    ids=sets.ids[v:v + nbat])

    def batched_shared(i):  # BB batches against one context's kb (a prefill's query batches)
        j, r = divmod(i, n_launch)
        nbat = min(BB, K - r * BB)
        v = (j * K + r * BB) % sets.n
        if v + nbat > sets.n:
            v = 0
        tbs.qsa_select_step_batched(sets.q32[v:v + nbat], sets.kb[v], w.n_kv, w.k, w.block,
                                    q16=sets.q16[v:v + nbat], scores=sets.scores[v:v + nbat],
                                    ids=sets.ids[v:v + nbat])

    def score_only(i):
        v = i % sets.n
        tbs.qsa_block_scores(sets.q16[v], sets.kb[v], w.n_kv, w.block, out=sets.scores[v])

    def select_only(i):
        v = i % sets.n
        tbs.qsa_select(sets.scores[v], w.k, out=sets.ids[v])

    def convert_only(i):
        v = i % sets.n
        tbs.qsa_f32_to_f16(sets.q32[v], out=sets.q16[v])

    with torch.cuda.stream(stream):
        for i in range(W):
            step(i)
    torch.cuda.synchronize()
    plan = tbs.qsa_arm().split("last call on this thread: ", 1)[-1]

    # CUDA graphs of exactly K calls each (captured once, replayed in turn
    # over all the rotating sets)
    replays = {name: rotating_replay(torch, stream, fn, cnt, n_sets) for name, fn, cnt, n_sets in
               (("step", step, K, sets.n), ("score", score_only, K, sets.n),
                ("select", select_only, K, sets.n), ("convert", convert_only, K, sets.n),
                ("batched", batched, n_launch, -(-sets.n // K) * n_launch),
                ("batched_shared", batched_shared, n_launch, -(-sets.n // K) * n_launch))}
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    step_ms = time_region(torch, stream, replays["step"], 5, args.min_timed_seconds, barrier if dist else None)
    clocks = sampler.stop()
    kern_ms = {name: statistics.median(time_region(torch, stream, replays[name], 5, 0.3))
               for name in ("score", "select", "convert")}
    batched_ms = time_region(torch, stream, replays["batched"], 5, 0.5, barrier if dist else None)
    shared_ms = time_region(torch, stream, replays["batched_shared"], 5, 0.5, barrier if dist else None)
    with torch.cuda.stream(stream):
        batched(0)
    torch.cuda.synchronize()
    batched_plan = tbs.qsa_arm().split("last call on this thread: ", 1)[-1]
    with torch.cuda.stream(stream):
        batched_shared(0)
    torch.cuda.synchronize()
    shared_plan = tbs.qsa_arm().split("last call on this thread: ", 1)[-1]

    ms_step = statistics.median(step_ms) / K
    value = aggregate_rate(world, units_per_step(w) * K, statistics.median(step_ms))

    # The step's roofline: one launch of the fused kernel (or, for a problem
    # too large for it, the chain of separate kernels, taken as a whole).
    # Algorithmic work per step: FLOPs of every block (2*nq*H*D*nb) and the
    # bytes each input and output moves once (f32 q read, kb read, scores
    # and ids written, plus the fp16 copy of q when the chain writes one).
    step_flops = 2.0 * w.nq * w.H * w.D * w.nb
    step_bytes = 4.0 * w.nq * w.H * w.D + 2.0 * w.nb * w.D + 4.0 * w.nq * w.nb + 4.0 * w.nq * w.k
    if with_q16:
        step_bytes += 2.0 * w.nq * w.H * w.D
    t_step = ms_step / 1e3
    t_flop = step_flops / (peaks["bf16_tflops"] * 1e12)
    t_byte = step_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_flop >= t_byte:
        roof = {"bound": "tensor", "achieved": step_flops / t_step / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": step_bytes / t_step / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if step_launches == 1:
        kname = plan.split(": ", 1)[-1].split(" ")[0]
        roof["traffic"] = traffic_for(kname, w)
        roof["kernel"] = f"{kname} (qsa_select_step: one launch per step)"
    else:
        roof["traffic"] = None
        roof["kernel"] = f"qsa_select_step as {step_launches} chained launches taken as one step"
    roof["plan"] = plan
    roof["peak_source"] = f"{peak_src} (fp16 dense taken equal to the measured bf16 burst)"
    roof["algorithmic"] = {"flops": step_flops, "bytes": step_bytes,
                           "t_roofline_us": max(t_flop, t_byte) * 1e6, "t_launch_us": t_step * 1e6}

    # the library's separate kernels, each timed alone (context)
    flops_score = 2.0 * w.nq * w.H * w.D * w.n_full
    bytes_score = 2.0 * w.nq * w.H * w.D + 2.0 * w.n_full * w.D + 4.0 * w.nq * w.nb
    bytes_select = 4.0 * w.nq * w.nb + 4.0 * w.nq * w.k
    bytes_convert = 6.0 * w.nq * w.H * w.D
    t = {n: kern_ms[n] / K / 1e3 for n in kern_ms}
    kernels = {
        "qsa_block_scores": {"us_per_launch": t["score"] * 1e6, "tflops": flops_score / t["score"] / 1e12,
                             "gbs": bytes_score / t["score"] / 1e9},
        "qsa_select": {"us_per_launch": t["select"] * 1e6, "gbs": bytes_select / t["select"] / 1e9},
        "qsa_f32_to_f16": {"us_per_launch": t["convert"] * 1e6, "gbs": bytes_convert / t["convert"] / 1e9},
    }

    # the same K batches, BB per launch (qsa_select_step_batched)
    t_b = statistics.median(batched_ms) / 1e3
    batched_res = {
        "batches_per_launch": BB, "launches": n_launch,
        "value": world * units_per_step(w) * K / t_b, "unit": UNIT,
        "ms_per_batch": t_b / K * 1e3,
        "roofline_frac": (K * max(t_flop, t_byte)) / t_b,
        "plan": batched_plan,
        "api": "qsa_select_step_batched with a kb per batch, q16 buffer given; CUDA graph of K/B "
               "calls",
    }
    t_s = statistics.median(shared_ms) / 1e3
    shared_res = {
        "batches_per_call": BB, "calls": n_launch,
        "value": world * units_per_step(w) * K / t_s, "unit": UNIT,
        "ms_per_batch": t_s / K * 1e3,
        "roofline_frac": (K * max(t_flop, t_byte)) / t_s,
        "plan": shared_plan,
        "api": "qsa_select_step_batched with one kb shared by the batches (a prefill's query "
               "batches against one context), q16 buffer given; CUDA graph of K/B calls",
    }

    # end-to-end through the host-buffer entry point
    e2e = run_e2e(torch, tbs, w, device, stream, K, W, barrier if dist else None, with_q16)

    launches_per_step = step_launches
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": workload_config(w, {
            "parallelism": f"replicas x{world} (independent query batches per GPU)",
            "l2": f"rotating {sets.n} distinct input/output sets ({sets.n * sets.per_set_bytes / 2**20:.0f} MiB > 2x L2)",
            "timing": f"CUDA graph of {K} steps; CUDA events on the launching stream; median of "
                      f"{len(step_ms)} repetitions",
            "accumulate": "fp32"}),
        "roofline": roof,
        "separate_kernels": kernels,
        "batched": batched_res,
        "batched_shared_kb": shared_res,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
    }
    if not args.no_per_config:
        res["per_config"] = run_per_config(
            torch, tbs, device, stream, peaks, peak_src, K, W,
            0.0 if args.no_cpu_baseline else args.per_config_cpu_seconds, barrier if dist else None)
    if not args.no_split:
        res["split_reduce"] = run_split(torch, tbs, device, stream, peaks, peak_src, K,
                                        barrier if dist else None)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def step_plan(tbs, w):
    """(with_q16, launches) of qsa_select_step on workload w: the fp16 query
    buffer is passed only where it changes the library's plan (large problems
    run the separate kernels, which need it)."""
    n0 = tbs.qsa_select_step_launches(w.nq, w.H, w.D, w.n_kv, w.k, w.block, with_q16=False)
    n1 = tbs.qsa_select_step_launches(w.nq, w.H, w.D, w.n_kv, w.k, w.block, with_q16=True)
    return (True, n1) if n1 != n0 else (False, n0)


def step_roofline(w, t_step, peaks, with_q16):
    """Roofline of one step of workload w measured at t_step seconds: the
    larger of its FLOP time at the fp16 tensor peak and its byte time at the
    HBM peak (algorithmic work: every block's FLOPs, each input read and each
    output written once, plus the fp16 query copy when the plan writes one)."""
    flops = 2.0 * w.nq * w.H * w.D * w.nb
    nbytes = 4.0 * w.nq * w.H * w.D + 2.0 * w.nb * w.D + 4.0 * w.nq * w.nb + 4.0 * w.nq * w.k
    if with_q16:
        nbytes += 2.0 * w.nq * w.H * w.D
    t_flop = flops / (peaks["bf16_tflops"] * 1e12)
    t_byte = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_flop >= t_byte:
        r = {"bound": "tensor", "achieved": flops / t_step / 1e12, "peak": peaks["bf16_tflops"],
             "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": nbytes / t_step / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["t_roofline_us"] = max(t_flop, t_byte) * 1e6
    r["flops"] = flops
    r["bytes"] = nbytes
    return r


PER_CONFIG = [w.name for w in qi.WORKLOADS + qi.DECODE_WORKLOADS]


def run_per_config(torch, tbs, device, stream, peaks, peak_src, K, W, cpu_budget, barrier):
    """Every workload and the decode shapes through qsa_select_step, each
    timed two ways: cold (a CUDA graph of K steps over rotating input/output
    sets larger than twice L2, so every step reads from HBM) and warm (K
    steps on one L2-resident set). Per entry: ms per step, query*blocks/s,
    the roofline of the cold number (and the warm one's fraction), and a
    bounded CPU-oracle sample (rank 0 of a one-rank job)."""
    from oracle import qsa_oracle as orc
    out = {}
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)

    def flush():  # write a buffer larger than L2, outside the timed region
        with torch.cuda.stream(stream):
            flush_buf.fill_(1.0)
    for name in PER_CONFIG:
        w = qi.BY_NAME[name]
        with_q16, launches = step_plan(tbs, w)
        # K distinct sets at most (each touched once per replay, after an L2
        # flush), or fewer large ones that add up to more than twice L2
        per = Sets.bytes_per_set(w)
        n_sets = min(K, max(3, math.ceil(2 * L2_BYTES / per)))
        sets = Sets(torch, tbs, w, device, n_sets * per, rank, max_distinct=8, min_sets=3)

        def step(i, sets=sets, w=w, with_q16=with_q16):
            v = i % sets.n
            tbs.qsa_select_step(sets.q32[v], sets.kb[v], w.n_kv, w.k, w.block,
                                q16=sets.q16[v] if with_q16 else None,
                                scores=sets.scores[v], ids=sets.ids[v])

        def step_warm(i, sets=sets, w=w, with_q16=with_q16):
            tbs.qsa_select_step(sets.q32[0], sets.kb[0], w.n_kv, w.k, w.block,
                                q16=sets.q16[0] if with_q16 else None,
                                scores=sets.scores[0], ids=sets.ids[0])

        with torch.cuda.stream(stream):
            for i in range(W):
                step(i)
        torch.cuda.synchronize()
        res = {}
        for label, fn in (("cold", step), ("warm", step_warm)):
            g = graph_of(torch, stream, fn, K)

            def rp(g=g):
                with torch.cuda.stream(stream):
                    g.replay()
            rp()
            torch.cuda.synchronize()
            ms = statistics.median(time_region(torch, stream, rp, 5, 0.25, barrier,
                                               pre=flush if label == "cold" else None))
            res[label] = ms / K
            del g
        t_cold = res["cold"] / 1e3
        t_warm = res["warm"] / 1e3
        roof = step_roofline(w, t_cold, peaks, with_q16)
        roof["peak_source"] = peak_src
        entry = {"nq": w.nq, "H": w.H, "D": w.D, "n_kv": w.n_kv, "nb": w.nb, "k": w.k,
                 "launches_per_step": launches,
                 "ms_per_step": res["cold"], "value": world * w.nq * w.nb / t_cold,
                 "unit": UNIT, "roofline": roof,
                 "warm": {"ms_per_step": res["warm"], "value": world * w.nq * w.nb / t_warm,
                          "roofline_frac": roof["t_roofline_us"] / 1e6 / t_warm},
                 "l2": f"cold: {sets.n} rotating sets ({sets.n * sets.per_set_bytes / 2**20:.0f} MiB); "
                       f"warm: one set"}
        if rank == 0 and world == 1 and cpu_budget > 0:
            entry["cpu_baseline"] = cpu_sample(orc, w, cpu_budget)
        out[name] = entry
        del sets
        torch.cuda.empty_cache()
    return out


def cpu_sample(orc, w, seconds):
    """The oracle on a bounded sample of workload w (whole batches when
    nq <= 256, else the first 256 queries), repeated for about `seconds`."""
    nq_s = min(w.nq, 256)
    q32, _ = qi.make_f32_inputs(w)
    _, kb = qi.make_inputs(w)
    n, t0 = 0, time.perf_counter()
    while n < 1 or time.perf_counter() - t0 < seconds:
        oracle_step(orc, w, q32, kb, nq_s)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n * nq_s * w.nb / dt, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} runs of {nq_s} of the {w.nq} queries in {dt:.1f} s"}


SPLIT_WORKLOAD = "split_g4_r8_c128_b2048"


def run_split(torch, tbs, device, stream, peaks, peak_src, K, barrier):
    """The second workload, the flash-attention decode split reduce
    (qsa_split_reduce), on its 128K-token shape: K calls in a CUDA graph over
    rotating input sets larger than twice L2, one shared workspace. HBM-bound:
    algorithmic bytes per call = partial_max + partial_sum + partial_out read
    once, out written once."""
    w = qi.SPLIT_BY_NAME[SPLIT_WORKLOAD]
    per_set = 8 * w.G * w.R * w.B + 2 * w.G * w.R * w.B * w.C + 4 * w.G * w.R * w.C
    n = max(4, -(-2 * L2_BYTES // per_set) + 1)
    base = [tuple(torch.from_numpy(a).to(device) for a in qi.make_split_partials(w, variant=v))
            for v in range(2)]
    sets = [base[v % 2] if v < 2 else tuple(t.clone() for t in base[v % 2]) for v in range(n)]
    outs = [torch.empty((w.G, w.R, w.C), dtype=torch.float32, device=device) for _ in range(n)]
    need = tbs.qsa_split_reduce_workspace_bytes(w.G, w.R, w.B, w.C)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=device)

    def call(i):
        pm, ps, po = sets[i % n]
        tbs.qsa_split_reduce(pm, ps, po, out=outs[i % n], workspace=ws)

    with torch.cuda.stream(stream):
        for i in range(4):
            call(i)
    torch.cuda.synchronize()
    g = graph_of(torch, stream, call, K)

    def replay():
        with torch.cuda.stream(stream):
            g.replay()
    replay()
    torch.cuda.synchronize()
    ms = time_region(torch, stream, replay, 5, 0.5, barrier)
    t = statistics.median(ms) / K / 1e3
    plan = tbs.qsa_arm().split("last call on this thread: ", 1)[-1]
    kname = plan.split(": ", 1)[-1].split(" ")[0]
    algo = 8.0 * w.G * w.R * w.B + 2.0 * w.G * w.R * w.B * w.C + 4.0 * w.G * w.R * w.C
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {
        "workload": w.name, "G": w.G, "R": w.R, "B": w.B, "C": w.C,
        "metric": "reduced (row, block) pairs/s", "value": world * w.G * w.R * w.B / t,
        "us_per_call": t * 1e6, "launches_per_call": 1,
        "roofline": {"bound": "hbm", "achieved": algo / t / 1e9, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": algo / t / 1e9 / peaks["hbm_gbs"],
                     "traffic": traffic_for(kname, w), "algorithmic_bytes": algo,
                     "peak_source": peak_src, "kernel": kname, "plan": plan},
        "l2": f"rotating {n} input sets ({n * per_set / 2**20:.0f} MiB > 2x L2)",
        "api": "qsa_split_reduce (CUDA graph of K calls)",
    }


E2E_STREAMS = int(os.environ.get("QSA_E2E_STREAMS", "6"))


def run_e2e(torch, tbs, w, device, stream, K, W, barrier, with_q16):
    """Same metric through HostStep (qsa_select_step_host_packed): each step
    copies its f32 queries and fp16 keys from one pinned host buffer (one
    copy), runs the step and copies the selected ids back (the step's result;
    the scores stay on the device). Steps go round-robin to E2E_STREAMS
    streams, each with its own device buffers, so one step's copies overlap
    another's kernel (the copy engines and the SMs work at once); two host
    input sets alternate; events on `stream` bracket all K steps (every
    stream joins it at the end)."""
    streams = [torch.cuda.Stream(device) for _ in range(E2E_STREAMS)]
    steps = [tbs.HostStep(w.nq, w.H, w.D, w.n_kv, w.k, w.block, device=device, with_q16=with_q16,
                          stream=streams[j]) for j in range(E2E_STREAMS)]
    inputs = []
    for v in range(2):
        q32, _ = qi.make_f32_inputs(w, variant=v)
        _, kb = qi.make_inputs(w, variant=v)
        buf = steps[0].new_input()
        steps[0].q32_view(buf).copy_(torch.from_numpy(q32))
        steps[0].kb_view(buf).copy_(torch.from_numpy(kb))
        inputs.append(buf)

    def one(i):
        steps[i % E2E_STREAMS](inputs[i % 2])

    def run(count):
        start = torch.cuda.Event()
        start.record(stream)
        for s_ in streams:
            s_.wait_event(start)
        for i in range(count):
            one(i)
        for s_ in streams:
            done = torch.cuda.Event()
            done.record(s_)
            stream.wait_event(done)

    run(W)
    torch.cuda.synchronize()
    ms = time_region(torch, stream, lambda: run(K), 3, 0.5, barrier)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    med = statistics.median(ms)
    return {"value": aggregate_rate(world, units_per_step(w) * K, med), "unit": UNIT,
            "h2d_bytes_per_step": w.nq * w.H * w.D * 4 + w.nb * w.D * 2,
            "d2h_bytes_per_step": w.nq * w.k * 4,
            "ms_per_step": med / K,
            "api": f"HostStep / qsa_select_step_host_packed (one pinned host buffer of f32 queries "
                   f"and fp16 keys in, the selected ids out; eager calls over {E2E_STREAMS} "
                   f"streams)"}


# --------------------------------------------------------------- CPU oracle
def oracle_step(orc, w, q32, kb, nq_sample=None):
    """The oracle as it stands on one batch (or its first nq_sample queries):
    fp16 conversion of q, float64 scores, the fp32 tail, lexsort top-k."""
    if nq_sample is not None:
        q32 = q32[:nq_sample]
    q16 = orc.f32_to_f16(q32)
    s = orc.scores_f64(q16, kb, w.n_kv, w.block)
    tail = orc.tail_scores_f32(q16, kb, w.n_kv, w.block)
    if tail is not None:
        s[:, -1] = tail
    return orc.select_topk(s, w.k)


def cpu_baseline(w, seconds):
    from oracle import qsa_oracle as orc
    q32, _ = qi.make_f32_inputs(w)
    _, kb = qi.make_inputs(w)
    oracle_step(orc, w, q32, kb)                  # warm
    n, t0 = 0, time.perf_counter()
    while n < 3 or time.perf_counter() - t0 < seconds:
        oracle_step(orc, w, q32, kb)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n * units_per_step(w) / dt, "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{n} whole {w.nq}-query batches of {w.name} in {dt:.1f} s (numpy float64 "
                      f"scores, fp32 tail, lexsort top-{w.k}; BLAS threads = all {os.cpu_count()} cores)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    from oracle import qsa_oracle as orc
    w = qi.BY_NAME[args.workload]
    K, W = args.steps, args.warmup
    nq_s = min(w.nq, 16)
    q32, _ = qi.make_f32_inputs(w)
    _, kb = qi.make_inputs(w)
    for _ in range(W):
        oracle_step(orc, w, q32, kb, nq_s)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_step(orc, w, q32, kb, nq_s)
    dt = time.perf_counter() - t0
    units = nq_s * w.nb
    value = units * K / dt
    sample = (f"each step: the first {nq_s} of the {w.nq} queries of {w.name} (numpy float64 "
              f"scores, fp32 tail, lexsort top-{w.k}); BLAS threads = all {os.cpu_count()} cores")
    res = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
           "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": workload_config(w, {"parallelism": "host cores (CPU oracle)"}),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
