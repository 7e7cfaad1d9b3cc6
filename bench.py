"""Benchmark of the split-K W4A16-g128 projection matmul on GB300.

One step = the seven Qwen3-4B projections (q, k, v, o, gate, up, down) at
M = 32 and M = 128 activation rows: 14 calls of qmm_w4a16_g128 with the
split chosen by the GB300 occupancy policy (each call = partition kernel +
reduce when it splits, one kernel when it does not).  Every call owns its
own weights; R rotating copies of the whole input set (more than twice the
L2 size together) make every step stream its weights from HBM.  Steps are
replayed as CUDA graphs; timing uses CUDA events on the launching stream.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the same workload instead.  Under torchrun each rank runs its own replica
(the matmul has no cross-GPU exchange); the job value is the max-over-ranks
time divided by all calls of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from split_w4a16_quantized_gb300 import inputs  # noqa: E402

METRIC = "µs/call and % of HBM/tensor roofline, W4A16-g128 split-K proj, M=16..2048"
UNIT = "us/call"
M_LIST = (32, 128)
PROJ = list(inputs.PROJECTIONS)
WORKLOAD = "Qwen3-4B projections q,k,v,o,gate,up,down (Kred->Nout) x M in {32,128}: " \
           "14 W4A16-g128 matmuls per step"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(M, Kred, Nout, split, partial_bytes=2):
    """Algorithmic bytes and flops of one call: packed weights, scales and
    biases, A, C, and the partial planes written and read back."""
    G = Kred // 128
    nbytes = Nout * Kred // 2 + 4 * Nout * G + 2 * M * Kred + 2 * M * Nout
    if split > 1:
        nbytes += 2 * partial_bytes * split * M * Nout
    return nbytes, 2.0 * M * Nout * Kred


def partition_algorithmic(M, Kred, Nout, split, partial_bytes=2):
    """Algorithmic bytes and flops of the partition kernel alone: packed
    weights, scales and biases, A, and the partial planes it writes."""
    G = Kred // 128
    nbytes = Nout * Kred // 2 + 4 * Nout * G + 2 * M * Kred + partial_bytes * split * M * Nout
    return nbytes, 2.0 * M * Nout * Kred


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the partition kernel, from one ncu capture per entry, keyed by the call and
# a hash of the kernel's sources at capture time: once the sources change the
# figure no longer describes the kernel and is reported as null.
NCU_TRAFFIC = {
    # python bench.py --only down:128 --launch-list --steps 1 --warmup 3 under
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
    # --clock-control none -k regex:w4a16_tc -s 2 -c 1: read + write
    ("down", 128, 4): (15789056, "dae890bb95cf3bea"),
    # the same with --partitions near-equal (split 7)
    ("down", 128, 7): (15788288, "8f0170d4d6878b62"),
    # the same for --only gate:32
    ("gate", 32, 2): (13461760, "8f0170d4d6878b62"),
}
TC_SOURCES = ("qmm_w4a16_tc.cu", "qmm_sm100.cuh", "qmm_device.cuh", "qmm_internal.h")
# The same for the decode-attention split kernel at the workload's planned
# split (python bench.py --attention-only --steps 2 --warmup 3 under
# ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
# --clock-control none -k regex:attn_split -s 3 -c 1), keyed by the split.
ATTN_TRAFFIC = {3: (670089728, "babc6b7daa2798ea")}
ATTN_SOURCES = ("qmm_attention.cu", "qmm_sm100.cuh", "qmm_device.cuh", "qmm_internal.h")


def tc_source_hash(sources=TC_SOURCES):
    import hashlib
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(ROOT, "split_w4a16_quantized_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def policy_desc():
    from split_w4a16_quantized_gb300 import qmm as Q
    parts = []
    for M in M_LIST:
        p = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        parts.append("M=%d: tile %dx%d, target_blocks %d, cap %d, min_k %d"
                     % (M, p.bm, p.bn, p.target_blocks, p.cap, p.min_k_per_split))
    return "GB300 preset (" + "; ".join(parts) + ")"


def roofline_time_s(nbytes, flops, peaks):
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    return (t_hbm, "hbm") if t_hbm >= t_tc else (t_tc, "tensor")


def step_roofline(wl, ms_per_step, peaks):
    """The whole step against its roofline: every call's algorithmic bytes
    (packed weights, scales and biases, A, C, and at split s > 1 the BF16
    planes written and read back) and flops, each call bounded by the slower
    of bytes at the measured HBM bandwidth and flops at the measured BF16
    peak; frac = the sum of those bounds / the measured step time."""
    nb = fl = t = 0.0
    for (_, M, Kred, Nout), s in zip(wl.calls, wl.split):
        b, f = algorithmic(M, Kred, Nout, s)
        nb, fl = nb + b, fl + f
        t += roofline_time_s(b, f, peaks)[0]
    us = ms_per_step * 1e3
    return {"bytes": int(nb), "flops": fl, "roofline_us": round(t * 1e6, 3),
            "us": round(us, 3), "frac": round(t * 1e6 / us, 4),
            "note": "per call: max(bytes / HBM, flops / BF16 peak), summed over the step"}


def max_over_ranks(ms: float, device=None) -> float:
    """The largest per-rank time (the job ends when the slowest rank ends)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value_us(ms_max: float, world: int, steps: int, ncalls: int) -> float:
    """Whole-job µs per call: the max-over-ranks time over every call of every rank."""
    return ms_max * 1e3 / (world * steps * ncalls)


ONLY = None  # (projection, M) when --only restricts the step to one call


def calls():
    if ONLY is not None:
        return [(ONLY[0], ONLY[1]) + inputs.PROJECTIONS[ONLY[0]]]
    return [(name, M) + inputs.PROJECTIONS[name] for M in M_LIST for name in PROJ]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        import atexit
        atexit.register(self._kill)
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(
                    (num(r[3]) for r in rows if num(r[3]) is not None), default=None)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Workload:
    """Device buffers for R rotating copies of the 14-call step."""

    def __init__(self, device, Q, l2_bytes, near_equal=False, split_req=0):
        self.Q = Q
        self.device = device
        self.split_req = split_req  # of every call of the step (0: the policy)
        self.calls = calls()
        self.host = []
        for name, M, Kred, Nout in self.calls:
            self.host.append(inputs.make_w4a16(M, Kred, Nout, seed=0))
        self.set_bytes = sum(p["A"].nbytes + p["Wq"].nbytes + p["scales"].nbytes +
                             p["biases"].nbytes for p in self.host)
        self.R = max(2, -(-2 * l2_bytes // self.set_bytes) + 1)
        first = [Q.to_device(p, device) for p in self.host]
        self.sets = [first] + [[{k: v.clone() for k, v in d.items()} for d in first]
                               for _ in range(self.R - 1)]
        self.C = [[torch.empty((M, Nout), dtype=torch.bfloat16, device=device)
                   for (_, M, _, Nout) in self.calls] for _ in range(self.R)]
        # split of each call under the partition rule in force, and under the
        # other rule (qmm_set_partitions); the near-equal one is never smaller
        self.split, self.split_alt = [], []
        ws_max = 16
        for (_, M, Kred, Nout) in self.calls:
            pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
            s_eq = Q.qmm_splitk_plan(M, Kred, Nout, pol)
            s_ne = Q.qmm_splitk_plan_near_equal(M, Kred, Nout, pol)
            if split_req:
                s_eq = s_ne = Q.qmm_call_plan(M, Kred, Nout, split_req)[0]
                ws_max = max(ws_max, Q.qmm_call_workspace_bytes(M, Kred, Nout, split_req))
            self.split.append(s_ne if near_equal else s_eq)
            self.split_alt.append(s_eq if near_equal else s_ne)
            ws_max = max(ws_max, Q.qmm_splitk_workspace_bytes(M, Nout, s_ne, Q.QMM_PARTIAL_BF16))
        # one workspace for every call, zeroed, with room beyond the largest
        # planes for the fused reduce's counter area (its last 32 KB), which
        # planes therefore never touch
        self.ws = torch.zeros(ws_max + (64 << 10), dtype=torch.uint8, device=device)

    def call(self, i, r, split_req=0):
        d = self.sets[r][i]
        return self.Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], self.C[r][i],
                                     split_req=split_req, workspace=self.ws)

    def step(self, r):
        for i in range(len(self.calls)):
            self.call(i, r, self.split_req)

    def launches_per_step(self):
        return sum(2 if s > 1 else 1 for s in self.split)


def graph_us_per_launch(fn, k, stream, reps=5):
    """Average µs per launch of fn(j), j = 0..k-1, captured back to back in one
    CUDA graph and replayed after warm-up: CUDA events on the launching
    stream around `reps` replays.  Each j uses its own copy of the inputs, and
    the k copies together exceed twice the L2 size, so every launch reads its
    weights from HBM while the kernels' code stays cached (as in a model's
    stream of calls)."""
    for j in range(k):
        fn(j)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            for j in range(k):
                fn(j)
    stream.wait_stream(cap)
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    del g
    return t0.elapsed_time(t1) * 1e3 / (reps * k)


def cold_copies(d, l2_bytes, keys=("A", "Wq", "scales", "biases")):
    """Enough copies of one call's inputs to exceed 2.2 x L2 (at least 4)."""
    nbytes = sum(d[k].numel() * d[k].element_size() for k in keys)
    k = max(4, -(-int(2.2 * l2_bytes) // nbytes))
    return [d] + [{key: d[key].clone() for key in keys} for _ in range(k - 1)]


def run_gpu(args, rank, world, local_rank):
    from split_w4a16_quantized_gb300 import build as qbuild
    qbuild.build()
    from split_w4a16_quantized_gb300 import qmm as Q
    import torch.distributed as dist

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    Q.qmm_set_kernels({"default": Q.QMM_KERNELS_DEFAULT, "mma": Q.QMM_KERNELS_MMA_SYNC,
                       "tc": Q.QMM_KERNELS_TCGEN05, "lean": Q.QMM_KERNELS_LEAN}[args.kernels])
    # the workload's weights are loaded once and never written by a kernel on
    # the stream, so the library may start weight work before the previous
    # kernel finishes (qmm_set_weights_static); --weights dynamic turns it off
    static_weights = args.weights == "static"
    Q.qmm_set_weights_static(static_weights)
    near_equal = args.partitions == "near-equal"
    rule = Q.QMM_PARTITIONS_NEAR_EQUAL if near_equal else Q.QMM_PARTITIONS_EQUAL
    alt_rule = Q.QMM_PARTITIONS_EQUAL if near_equal else Q.QMM_PARTITIONS_NEAR_EQUAL
    Q.qmm_set_partitions(rule)
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    sms = props.multi_processor_count
    peaks, peak_src = load_peaks()
    wl = Workload(device, Q, l2, near_equal,
                  {"policy": 0, "planned": Q.QMM_SPLIT_PLANNED,
                   "balanced": Q.QMM_SPLIT_BALANCED}[args.split_req])
    stream = torch.cuda.current_stream()
    step = wl.step
    if args.grouped:  # profiling aid: the step's calls as one grouped call
        Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_PERSISTENT if args.grouped == "persistent"
                                   else Q.QMM_GROUPED_TILES)
        if args.group_plan:
            Q.qmm_set_group_plan(Q.QMM_GROUP_PLAN_GROUP)
        g_arrays = [Q.group_calls([dict(wl.sets[r][i], C=wl.C[r][i])
                                   for i in range(len(wl.calls))]) for r in range(wl.R)]
        g_ws = torch.zeros(max(Q.qmm_group_workspace_bytes(g_arrays[0]), 16), dtype=torch.uint8,
                           device=device)
        step = lambda r: Q.qmm_w4a16_g128_grouped(g_arrays[r], g_ws)

    # warm-up: eager step per set (first calls set kernel attributes), then graphs
    for r in range(wl.R):
        step(r)
    torch.cuda.synchronize()
    graphs = []
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for r in range(wl.R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step(r)
            graphs.append(g)
    stream.wait_stream(cap)
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank).start() if not args.launch_list else None
    if clocks:
        time.sleep(0.3)
    for k in range(args.warmup):
        graphs[k % wl.R].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        graphs[k % wl.R].replay()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(t0.elapsed_time(t1), device)

    if args.launch_list:
        launches, splits = None, wl.split
        if args.grouped:
            widths = len({Q.qmm_kernel_tile(M)[0] for (_, M, _, _) in wl.calls})
            splits = Q.qmm_group_plan([(M, K, N) for (_, M, K, N) in wl.calls]) \
                if args.group_plan else wl.split
            launches = widths + (1 if any(sp > 1 for sp in splits) else 0)
        return {"ms": ms, "wl": wl, "launch_list": True, "grouped_launches": launches,
                "splits": splits}

    def time_variant(setter, value):
        """The step re-captured with one library switch changed, same timing."""
        prev = setter(value)
        gs = []
        with torch.cuda.stream(cap):
            for r in range(wl.R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    wl.step(r)
                gs.append(g)
        setter(prev)
        torch.cuda.synchronize()
        for k in range(args.warmup):
            gs[k % wl.R].replay()
        t0.record(stream)
        for k in range(args.steps):
            gs[k % wl.R].replay()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    # the same step with programmatic dependent launch off, and with the
    # static-weights promise flipped, for comparison
    ms_nopdl = time_variant(Q.qmm_set_pdl, False)
    ms_wflip = time_variant(Q.qmm_set_weights_static, not static_weights)
    ms_fused = time_variant(Q.qmm_set_reduce, Q.QMM_REDUCE_FUSED)
    ms_cluster = time_variant(Q.qmm_set_reduce, Q.QMM_REDUCE_CLUSTER)
    ms_alt = time_variant(Q.qmm_set_partitions, alt_rule)

    # the same 14 calls as one grouped call per step (qmm_w4a16_g128_grouped):
    # one partition launch per tile width and one reduce launch
    group_arrays = [Q.group_calls([dict(wl.sets[r][i], C=wl.C[r][i])
                                   for i in range(len(wl.calls))]) for r in range(wl.R)]
    gws = torch.zeros(max(Q.qmm_group_workspace_bytes(group_arrays[0]), 16), dtype=torch.uint8,
                      device=device)

    def time_grouped(ws=gws):
        gs = []
        with torch.cuda.stream(cap):
            for r in range(wl.R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    Q.qmm_w4a16_g128_grouped(group_arrays[r], ws)
                gs.append(g)
        torch.cuda.synchronize()
        for k in range(args.warmup):
            gs[k % wl.R].replay()
        t0.record(stream)
        for k in range(args.steps):
            gs[k % wl.R].replay()
        t1.record(stream)
        torch.cuda.synchronize()
        del gs
        return t0.elapsed_time(t1)
    ms_grouped = time_grouped()  # the library's default schedule (persistent)
    # the same grouped step with one CTA per tile in every launch
    prev_sched = Q.qmm_set_grouped_schedule(Q.QMM_GROUPED_TILES)
    ms_grouped_tiles = time_grouped()
    Q.qmm_set_grouped_schedule(prev_sched)
    # and with splits planned for the group (qmm_set_group_plan)
    prev_plan = Q.qmm_set_group_plan(Q.QMM_GROUP_PLAN_GROUP)
    plan_ws = torch.zeros(max(Q.qmm_group_workspace_bytes(group_arrays[0]), 16),
                          dtype=torch.uint8, device=device)
    ms_grouped_plan = time_grouped(plan_ws)
    group_plan_splits = Q.qmm_group_plan([(M, Kred, Nout) for (_, M, Kred, Nout) in wl.calls])
    Q.qmm_set_group_plan(prev_plan)
    del plan_ws
    tile_widths = len({Q.qmm_kernel_tile(M)[0] for (_, M, _, _) in wl.calls})
    grouped_launches = tile_widths + (1 if any(s > 1 for s in wl.split) else 0)

    # per call: policy split vs the unsplit control, each timed as a graph of
    # back-to-back launches over copies of its inputs larger than L2.  These and
    # the roofline's kernel timing run without the static-weights early start:
    # back to back, a call whose grid leaves SMs free would otherwise overlap
    # the next identical call, which measures the overlap, not the kernel
    Q.qmm_set_weights_static(False)
    per_call = []
    dom = None
    for i, (name, M, Kred, Nout) in enumerate(wl.calls):
        s = wl.split[i]
        cps = cold_copies(wl.sets[0][i], l2)
        C = wl.C[0][i]

        def call(j, split_req):
            d = cps[j]
            Q.qmm_w4a16_g128(d["A"], d["Wq"], d["scales"], d["biases"], C, split_req=split_req,
                             workspace=wl.ws)
        us_s = graph_us_per_launch(lambda j: call(j, 0), len(cps), stream)
        us_1 = graph_us_per_launch(lambda j: call(j, 1), len(cps), stream) if s > 1 else us_s
        s_alt = wl.split_alt[i]
        if s_alt != s:
            Q.qmm_set_partitions(alt_rule)
            us_alt = graph_us_per_launch(lambda j: call(j, 0), len(cps), stream)
            Q.qmm_set_partitions(rule)
        else:
            us_alt = us_s
        nb_alt, fl_alt = algorithmic(M, Kred, Nout, s_alt)
        t_roof_alt, _ = roofline_time_s(nb_alt, fl_alt, peaks)
        alt = "equal" if near_equal else "near_equal"
        nb, fl = algorithmic(M, Kred, Nout, s)
        nb1, _ = algorithmic(M, Kred, Nout, 1)
        t_roof, bound = roofline_time_s(nb, fl, peaks)
        t_roof1, _ = roofline_time_s(nb1, fl, peaks)
        per_call.append({"proj": name, "M": M, "Kred": Kred, "Nout": Nout, "split": s,
                         "us_split": round(us_s, 3), "us_unsplit": round(us_1, 3),
                         "bytes": nb, "flops": fl, "bound": bound,
                         "roof_frac_split": round(t_roof * 1e6 / us_s, 4),
                         "roof_frac_unsplit": round(t_roof1 * 1e6 / us_1, 4),
                         "tbps_split": round(nb / us_s / 1e6, 3),
                         "tflops_split": round(fl / us_s / 1e6, 2),
                         "split_" + alt: s_alt, "us_" + alt: round(us_alt, 3),
                         "roof_frac_" + alt: round(t_roof_alt * 1e6 / us_alt, 4),
                         "copies": len(cps)})
        if dom is None or us_s > per_call[dom["index"]]["us_split"]:
            dom = {"index": i, "split": s}
            # the call's partition kernel on its own (the roofline's kernel) and
            # its reduce, timed the same way
            if s > 1:
                planes = wl.ws[:s * M * Nout * 2].view(torch.bfloat16).view(s, M, Nout)

                def part(j):
                    d = cps[j]
                    Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"],
                                               planes, s)
                dom["us_partition"] = graph_us_per_launch(part, len(cps), stream)
                dom["us_reduce"] = graph_us_per_launch(
                    lambda j: Q.qmm_splitk_reduce(planes, Q.QMM_PARTIAL_BF16, s, M, Nout, C),
                    len(cps), stream)
            # and under the other partition rule, when that splits it otherwise
            if s_alt > 1 and s_alt != s:
                planes_alt = wl.ws[:s_alt * M * Nout * 2].view(torch.bfloat16).view(s_alt, M, Nout)

                def part_alt(j):
                    d = cps[j]
                    Q.qmm_w4a16_g128_partition(d["A"], d["Wq"], d["scales"], d["biases"],
                                               planes_alt, s_alt)
                Q.qmm_set_partitions(alt_rule)
                dom["split_alt"] = s_alt
                dom["us_partition_alt"] = graph_us_per_launch(part_alt, len(cps), stream)
                Q.qmm_set_partitions(rule)
        del cps
    prefill = prefill_sweep(Q, device, stream, l2, peaks) if rank == 0 else None
    sweep = shape_sweep(Q, device, stream, l2, peaks) if rank == 0 else None
    Q.qmm_set_weights_static(static_weights)
    sample = clocks.stop()
    dense = dense_sweep(Q, device, stream, sms, l2) if rank == 0 else None
    e2e = run_e2e(wl, Q, device, stream, min(args.steps, 20))
    e2e_resident = run_e2e(wl, Q, device, stream, min(args.steps, 20), weights_resident=True)
    e2e_resident_graph = run_e2e(wl, Q, device, stream, min(args.steps, 20),
                                 weights_resident=True, graphed=True)
    overlap = overlap_sweep(wl, Q, device) if rank == 0 else None
    attention = attention_bench(Q, device, stream, peaks, l2) if rank == 0 else None
    return {"ms": ms, "ms_nopdl": ms_nopdl, "ms_wflip": ms_wflip, "ms_fused": ms_fused, "ms_cluster": ms_cluster,
            "ms_alt": ms_alt, "ms_grouped": ms_grouped,
            "ms_grouped_tiles": ms_grouped_tiles, "ms_grouped_plan": ms_grouped_plan,
            "group_plan_splits": group_plan_splits, "grouped_launches": grouped_launches,
            "per_call": per_call, "dom": dom,
            "clocks": sample, "wl": wl,
            "peaks": peaks,
            "peak_src": peak_src, "l2": l2, "sms": sms, "dense": dense, "e2e": e2e,
            "e2e_resident": e2e_resident, "e2e_resident_graph": e2e_resident_graph,
            "prefill": prefill, "sweep": sweep, "overlap": overlap, "attention": attention}


def prefill_sweep(Q, device, stream, l2, peaks):
    """The prefill regime (M = 2048) of each projection shape: the policy's
    split (the unsplit kernel wherever the base grid already fills the GPU),
    graphs of back-to-back calls over input copies larger than L2, tensor
    throughput against the measured dense BF16 peak.  Where the balanced
    split (QMM_SPLIT_BALANCED) plans the call otherwise -- head rows cut off
    a partial last wave, or the narrower tile where the wide one has no full
    wave -- its head rows, tile, split (of the tail) and time are given
    beside it."""
    out = []
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=device)
    for name in PROJ:
        Kred, Nout = inputs.PROJECTIONS[name]
        M = 2048
        d = Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=0), device)
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        split = Q.qmm_splitk_plan(M, Kred, Nout, pol)
        cps = cold_copies(d, l2)
        C = torch.empty((M, Nout), dtype=torch.bfloat16, device=device)

        def call(j, req=0):
            c = cps[j]
            Q.qmm_w4a16_g128(c["A"], c["Wq"], c["scales"], c["biases"], C, split_req=req,
                             workspace=ws)
        us = graph_us_per_launch(call, len(cps), stream)
        fl = 2.0 * M * Nout * Kred
        bm, bn = Q.qmm_kernel_tile(M)
        row = {"proj": name, "M": M, "split": split,
               "ctas": -(-M // bm) * -(-Nout // bn) * split, "us": round(us, 3),
               "tflops": round(fl / us / 1e6, 1),
               "frac_of_bf16_peak": round(fl / us / 1e6 / peaks["bf16_tflops"], 3)}
        s_b, bm_b, bn_b, head = Q.qmm_call_plan(M, Kred, Nout, Q.QMM_SPLIT_BALANCED,
                                                with_head=True)
        if head > 0 or (bm_b, bn_b) != (bm, bn):
            us_b = graph_us_per_launch(lambda j: call(j, Q.QMM_SPLIT_BALANCED), len(cps), stream)
            row["balanced"] = {"head_rows": head, "tile": [bm_b, bn_b], "split": s_b,
                               "us": round(us_b, 3),
                               "tflops": round(fl / us_b / 1e6, 1),
                               "frac_of_bf16_peak": round(fl / us_b / 1e6 / peaks["bf16_tflops"],
                                                          3)}
        out.append(row)
        del cps, d
    return out


def shape_sweep(Q, device, stream, l2, peaks):
    """The policy's split against its control on every shape of the workload
    configs that the 14-call step does not hold:
    - the M = 16 K-projection (the small case);
    - M in {16, 64} on the seven projections;
    - the ragged shape (Kred 2560, Nout 1000) at M in {16, 32, 64, 128, 2048};
    - M = 2048 on the seven projections;
    - the decode regime, M in {1, 4, 8} on k, o and down (the policy then keeps
      at least 512 reduction elements per partition).
    The control is the unsplit kernel where the policy splits.  Where the
    policy keeps the unsplit kernel because the base grid fills the GPU, the
    control is a forced split of 2, so the row shows whether not splitting was
    the faster choice.  Each side is a graph of back-to-back calls over input
    copies larger than L2, without the static-weights early start."""
    shapes = []
    for M in (16, 64, 2048):
        shapes += [(name, M) for name in PROJ]
    shapes += [("ragged", M) for M in (16, 32, 64, 128, 2048)]
    shapes += [(name, M) for M in (1, 4, 8) for name in ("k", "o", "down")]
    rows = []
    for name, M in shapes:
        Kred, Nout = inputs.RAGGED if name == "ragged" else inputs.PROJECTIONS[name]
        d = Q.to_device(inputs.make_w4a16(M, Kred, Nout, seed=0), device)
        pol = Q.qmm_policy_preset(Q.QMM_PRESET_GB300, M)
        split = Q.qmm_splitk_plan(M, Kred, Nout, pol)
        control = 1 if split > 1 else 2
        planned = Q.qmm_group_plan([(M, Kred, Nout)])[0]  # QMM_SPLIT_PLANNED's split
        ws = torch.empty(max(16, Q.qmm_splitk_workspace_bytes(M, Nout, max(split, control, planned),
                                                               Q.QMM_PARTIAL_BF16)),
                         dtype=torch.uint8, device=device)
        cps = cold_copies(d, l2)
        C = torch.empty((M, Nout), dtype=torch.bfloat16, device=device)

        def call(j, split_req):
            c = cps[j]
            Q.qmm_w4a16_g128(c["A"], c["Wq"], c["scales"], c["biases"], C,
                             split_req=split_req, workspace=ws)
        us = graph_us_per_launch(lambda j: call(j, 0), len(cps), stream)
        us_c = graph_us_per_launch(lambda j: call(j, control), len(cps), stream)
        us_p = graph_us_per_launch(lambda j: call(j, Q.QMM_SPLIT_PLANNED), len(cps), stream) \
            if planned != split else None
        nb, fl = algorithmic(M, Kred, Nout, split)
        t_roof, bound = roofline_time_s(nb, fl, peaks)
        bm, bn = Q.qmm_kernel_tile(M)
        rows.append({"proj": name, "M": M, "Kred": Kred, "Nout": Nout, "split": split,
                     "base_ctas": -(-M // bm) * -(-Nout // bn), "us": round(us, 3),
                     "control_split": control, "control_us": round(us_c, 3),
                     "speedup_vs_control": round(us_c / us, 3), "bound": bound,
                     "roofline_frac": round(t_roof * 1e6 / us, 4),
                     "planned_split": planned,
                     "planned_us": round(us_p, 3) if us_p is not None else None})
        del cps, d, ws
    split_rows = [r for r in rows if r["split"] > 1]
    kept = [r for r in rows if r["split"] == 1]
    differ = [r for r in rows if r["planned_us"] is not None]
    summary = {"shapes": len(rows), "policy_splits": len(split_rows),
               "split_beats_unsplit": sum(r["us"] < r["control_us"] for r in split_rows),
               "policy_unsplit": len(kept),
               "unsplit_beats_split_2": sum(r["us"] < r["control_us"] for r in kept),
               "planned_differs": len(differ),
               "planned_faster": sum(r["planned_us"] < r["us"] for r in differ)}
    return {"summary": summary, "rows": rows}


def dense_sweep(Q, device, stream, sms, l2):
    """Dense BF16 split-K GEMM 512 x 512 x 16384 (128 x 128 tiles) over the
    split counts of the one-wave / two-wave model; graphs of back-to-back
    launches over input copies larger than L2, CUDA events."""
    d = inputs.make_dense(512, 512, 16384, seed=0)
    f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    cps = cold_copies({"A": f(d["A"]), "W": f(d["W"])}, l2, keys=("A", "W"))
    C = torch.empty((512, 512), dtype=torch.bfloat16, device=device)
    ws = torch.empty(Q.qmm_gemm_workspace_bytes(512, 512, 16), dtype=torch.uint8, device=device)
    out = []
    for s in (1, 2, 4, 6, 8, 9, 12, 16):
        us = graph_us_per_launch(
            lambda j: Q.qmm_gemm_bf16_splitk(cps[j]["A"], cps[j]["W"], C, s, ws), len(cps),
            stream)
        out.append({"split": s, "blocks": 16 * s, "waves": -(-16 * s // sms), "us": round(us, 3),
                    "tflops": round(2 * 512 * 512 * 16384 / us / 1e6, 2)})
    return out


def attention_bench(Q, device, stream, peaks, l2):
    """Split-KV decode attention (qmm_decode_attention) on the Qwen3-4B heads
    (32 query, 8 KV, dim 128): 32 sequences with lengths mixed uniformly in
    [1024, 8192].  The KV history (about 0.6 GB) is far larger than L2, so
    each call reads it from HBM.  Timed as a graph of back-to-back calls, for
    the plan's split and a few forced ones; the roofline is the HBM copy
    bandwidth over the bytes a call must move (the valid K and V rows, q, O
    and, when split, the partial states written and read back)."""
    h = inputs.ATTENTION_HEADS
    B, Lmax = 32, 8192
    prob = inputs.make_attention(B, h["Hq"], h["Hkv"], Lmax, h["D"], seed=0, lmin=1024)
    d = Q.attention_to_device(prob, device)
    O = torch.empty((B, h["Hq"], h["D"]), dtype=torch.bfloat16, device=device)
    plan = Q.qmm_decode_attention_splits(B, h["Hq"], h["Hkv"], Lmax)
    ws = torch.empty(max(Q.qmm_decode_attention_workspace_bytes(B, h["Hq"], h["D"], 16), 16),
                     dtype=torch.uint8, device=device)
    kv_bytes = int(prob["lens"].sum()) * h["Hkv"] * h["D"] * 2 * 2
    qo_bytes = 2 * B * h["Hq"] * h["D"] * 2
    out = {"workload": "Qwen3-4B heads (Hq 32, Hkv 8, D 128), B=32, lens U[1024, 8192] "
                       "(seed 0), K/V BF16 head-major",
           "kv_bytes": kv_bytes, "plan_split": plan, "splits": []}
    calls_per_graph = max(4, -(-3 * l2 // kv_bytes))
    for S in sorted({plan, 1, 2, 4, 8, 16}):
        us = graph_us_per_launch(
            lambda j: Q.qmm_decode_attention(d["q"], d["K"], d["V"], d["lens"], O,
                                             splits_req=S, workspace=ws),
            calls_per_graph, stream)
        part = 2 * B * h["Hq"] * S * (h["D"] + 2) * 4 if S > 1 else 0
        nbytes = kv_bytes + qo_bytes + part
        gbs = nbytes / us / 1e3
        out["splits"].append({"split": S, "ctas": S * B * h["Hkv"], "us": round(us, 3),
                              "gbs": round(gbs, 1),
                              "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)})
    best = min(out["splits"], key=lambda r: r["us"])
    out["plan"] = next(r for r in out["splits"] if r["split"] == plan)
    out["best"] = best
    # ncu DRAM bytes of one launch of the split kernel at the plan's split,
    # while the kernel's sources are the ones captured (else null)
    tr = ATTN_TRAFFIC.get(plan)
    out["plan"]["traffic"] = tr[0] if tr and tr[1] == tc_source_hash(ATTN_SOURCES) else None
    return out


def run_attention_only(args):
    """--attention-only: W warm-up and K timed decode-attention calls of the
    bench's attention workload at the plan's split, one JSON line."""
    from split_w4a16_quantized_gb300 import build as qbuild
    qbuild.build()
    from split_w4a16_quantized_gb300 import qmm as Q
    device = torch.device("cuda", 0)
    h = inputs.ATTENTION_HEADS
    B, Lmax = 32, 8192
    prob = inputs.make_attention(B, h["Hq"], h["Hkv"], Lmax, h["D"], seed=0, lmin=1024)
    d = Q.attention_to_device(prob, device)
    O = torch.empty((B, h["Hq"], h["D"]), dtype=torch.bfloat16, device=device)
    S = Q.qmm_decode_attention_splits(B, h["Hq"], h["Hkv"], Lmax)
    ws = torch.empty(max(Q.qmm_decode_attention_workspace_bytes(B, h["Hq"], h["D"], S), 16),
                     dtype=torch.uint8, device=device)
    run = lambda: Q.qmm_decode_attention(d["q"], d["K"], d["V"], d["lens"], O, workspace=ws)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        run()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"attention_only": True, "split": S, "calls": args.steps,
                      "us_per_call": round(t0.elapsed_time(t1) * 1e3 / args.steps, 3),
                      "status": Q.qmm_kernel_status(clear=True)}), flush=True)


def run_dense_only(args):
    """--dense-only S: W warm-up and K timed calls of the dense BF16 split-K
    GEMM 512 x 512 x 16384 at split S (the partition kernel and the reduce),
    one JSON line.  A profiling aid: one copy of the inputs (they stay in L2)."""
    from split_w4a16_quantized_gb300 import build as qbuild
    qbuild.build()
    from split_w4a16_quantized_gb300 import qmm as Q
    device = torch.device("cuda", 0)
    d = inputs.make_dense(512, 512, 16384, seed=0)
    f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    A, W = f(d["A"]), f(d["W"])
    C = torch.empty((512, 512), dtype=torch.bfloat16, device=device)
    ws = torch.empty(Q.qmm_gemm_workspace_bytes(512, 512, 16), dtype=torch.uint8, device=device)
    run = lambda: Q.qmm_gemm_bf16_splitk(A, W, C, args.dense_only, ws)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        run()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"dense_only": True, "split": args.dense_only, "calls": args.steps,
                      "us_per_call": round(t0.elapsed_time(t1) * 1e3 / args.steps, 3),
                      "status": Q.qmm_kernel_status(clear=True)}), flush=True)


def overlap_sweep(wl, Q, device, reps=10):
    """The copy-in / compute / copy-out pipeline (qmm_w4a16_g128_stream) on the
    step's 14 calls: activations from pinned host memory, weights resident,
    outputs back to pinned host memory.  Per-chunk engine times are measured
    engine by engine (each engine's 14 chunks back to back on one stream,
    events between chunks); the pipeline's end-to-end time is measured for 1,
    2 and 3 buffers on three streams and set beside the schedule model's
    prediction from the measured engine times (qmm_overlap_schedule, output
    buffers reused as the executor does).  Every timed sequence is enqueued
    behind a short device-side delay (torch.cuda._sleep, a bounded clock
    loop), so the GPU runs it back to back instead of at the host's launch
    pace."""
    n = len(wl.calls)
    chunks = []
    for p, d in zip(wl.host, wl.sets[0]):
        M, Nout = p["A"].shape[0], p["Wq"].shape[0]
        chunks.append({"A": torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16)
                       .pin_memory(),
                       "C": torch.empty((M, Nout), dtype=torch.bfloat16).pin_memory(),
                       "Wq": d["Wq"], "scales": d["scales"], "biases": d["biases"],
                       "A_dev": d["A"]})
    calls = Q.stream_calls(chunks)
    s_in, s_comp, s_out = (torch.cuda.Stream(device=device) for _ in range(3))
    arena = torch.zeros(Q.qmm_stream_arena_bytes(calls, 3), dtype=torch.uint8, device=device)
    C_dev = [torch.empty_like(c["C"], device=device) for c in chunks]

    hold = int(2e-3 * 2.0e9)  # about 2 ms of SM clocks: time to enqueue a sequence

    def engine_times(enqueue, st):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        acc = np.zeros(n)
        for r in range(reps + 2):
            with torch.cuda.stream(st):
                torch.cuda._sleep(hold)
                ev[0].record(st)
                for i in range(n):
                    enqueue(i)
                    ev[i + 1].record(st)
            st.synchronize()
            if r >= 2:
                acc += [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(n)]
        return acc / reps

    t_load = engine_times(lambda i: chunks[i]["A_dev"].copy_(chunks[i]["A"], non_blocking=True),
                          s_in)
    t_comp = engine_times(lambda i: Q.qmm_w4a16_g128(
        chunks[i]["A_dev"], chunks[i]["Wq"], chunks[i]["scales"], chunks[i]["biases"], C_dev[i],
        workspace=wl.ws, stream=s_comp), s_comp)
    t_store = engine_times(lambda i: chunks[i]["C"].copy_(C_dev[i], non_blocking=True), s_out)
    out = {"chunks": n, "engine_us_per_step": {"load": round(float(t_load.sum()), 2),
                                               "compute": round(float(t_comp.sum()), 2),
                                               "store": round(float(t_store.sum()), 2)},
           "measured_us": {}, "model_us": {}}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for b in (1, 2, 3):
        total = 0.0
        for r in range(reps + 2):
            with torch.cuda.stream(s_in):
                torch.cuda._sleep(hold)
            t0.record(s_in)
            Q.qmm_w4a16_g128_stream(calls, b, arena, s_in, s_comp, s_out)
            t1.record(s_out)
            torch.cuda.synchronize()
            if r >= 2:
                total += t0.elapsed_time(t1) * 1e3
        out["measured_us"][str(b)] = round(total / reps, 2)
        out["model_us"][str(b)] = round(Q.qmm_overlap_schedule(n, b, t_load, t_comp, t_store,
                                                                out_reuse=True), 2)
    out["speedup_2_buffers"] = {"measured": round(out["measured_us"]["1"] /
                                                  out["measured_us"]["2"], 3),
                                "model": round(out["model_us"]["1"] / out["model_us"]["2"], 3)}
    out["note"] = ("weights resident; per chunk the activations come in and the output goes "
                   "out through pinned host memory; reps=%d" % reps)
    return out


def run_e2e(wl, Q, device, stream, steps, weights_resident=False, graphed=False):
    """The same step through the public API with host buffers: per step the
    pinned-host inputs of all 14 calls (A, packed weights, scales, biases) are
    copied in, the calls run, and every output is copied back, all inside the
    timed region.  Inputs and outputs of a step are packed into one pinned
    buffer each (one host-to-device and one device-to-host copy per step);
    copy streams move step k+1's inputs in and step k-1's outputs out while
    step k computes (two device input and output buffers, ordered by events).
    weights_resident: the packed weights, scales and biases are uploaded once
    before the timed region, as a deployed model's are, and only the
    activations move in.  graphed: each buffer set's 14 public-API calls are
    captured once in a CUDA graph and a step replays it (one host call instead
    of 14)."""
    keys = ("A",) if weights_resident else ("A", "Wq", "scales", "biases")
    resident = [Q.to_device(p, device) for p in wl.host] if weights_resident else None
    align = lambda n: (n + 255) // 256 * 256
    in_off, out_off, ni, no = [], [], 0, 0
    for p, (_, M, _, Nout) in zip(wl.host, wl.calls):
        offs = {}
        for k in keys:
            offs[k] = ni
            ni += align(p[k].nbytes)
        in_off.append(offs)
        out_off.append(no)
        no += align(M * Nout * 2)
    host_in = torch.empty(ni, dtype=torch.uint8).pin_memory()
    hv = host_in.numpy()
    for p, offs in zip(wl.host, in_off):
        for k in keys:
            raw = np.ascontiguousarray(p[k]).view(np.uint8).reshape(-1)
            hv[offs[k]:offs[k] + raw.size] = raw
    host_out = torch.empty(no, dtype=torch.uint8).pin_memory()
    dev_in = [torch.empty(ni, dtype=torch.uint8, device=device) for _ in range(2)]
    dev_out = [torch.empty(no, dtype=torch.uint8, device=device) for _ in range(2)]

    def views(buf, obuf):
        calls = []
        for i, (p, offs, oo, (_, M, Kred, Nout)) in enumerate(
                zip(wl.host, in_off, out_off, wl.calls)):
            t = dict(resident[i]) if resident else {}
            for k, dt in zip(keys, (torch.bfloat16, torch.int32, torch.bfloat16, torch.bfloat16)):
                n = p[k].nbytes
                t[k] = buf[offs[k]:offs[k] + n].view(dt).view(p[k].shape)
            t["C"] = obuf[oo:oo + M * Nout * 2].view(torch.bfloat16).view(M, Nout)
            calls.append(t)
        return calls
    sets = [views(dev_in[b], dev_out[b]) for b in range(2)]

    def calls(b):
        for t in sets[b]:
            Q.qmm_w4a16_g128(t["A"], t["Wq"], t["scales"], t["biases"], t["C"],
                             workspace=wl.ws)

    graphs = None
    if graphed:
        cap = torch.cuda.Stream(device=device)
        cap.wait_stream(stream)
        graphs = []
        with torch.cuda.stream(cap):
            for b in range(2):
                calls(b)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    calls(b)
                graphs.append(g)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
    # two copy streams, each moving half of a step's inputs (two copy engines),
    # and one stream for the outputs, so that a step's D2H copy overlaps the
    # next step's calls
    copies = [torch.cuda.Stream(device=device) for _ in range(2)]
    out_copy = torch.cuda.Stream(device=device)
    half = ni // 2 // 256 * 256
    parts = [(0, half), (half, ni)]
    in_ready = [[torch.cuda.Event() for _ in range(2)] for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    issue = [0.0]

    def run(nsteps):
        for k in range(nsteps):
            b = k % 2
            for c, (lo, hi) in zip(copies, parts):
                with torch.cuda.stream(c):
                    if k >= 2:
                        c.wait_event(in_free[b])
                    dev_in[b][lo:hi].copy_(host_in[lo:hi], non_blocking=True)
            for c, ev in zip(copies, in_ready[b]):
                ev.record(c)
                stream.wait_event(ev)
            if k >= 2:
                stream.wait_event(out_done[b])
            t0 = time.perf_counter()
            if graphs is not None:
                graphs[b].replay()
            else:
                calls(b)
            issue[0] += time.perf_counter() - t0
            in_free[b].record(stream)
            computed[b].record(stream)
            with torch.cuda.stream(out_copy):
                out_copy.wait_event(computed[b])
                host_out.copy_(dev_out[b], non_blocking=True)
                out_done[b].record(out_copy)
        for c in copies + [out_copy]:
            c.synchronize()
        stream.synchronize()

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for c in copies + [out_copy]:
        c.wait_stream(stream)
    issue[0] = 0.0
    run(steps)
    for c in copies + [out_copy]:
        stream.wait_stream(c)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(p[k].nbytes for p in wl.host for k in keys)
    d2h = sum(M * Nout * 2 for (_, M, _, Nout) in wl.calls)
    return {"value": round(ms * 1e3 / len(wl.calls), 3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "h2d_gbps": round(h2d / (ms * 1e-3) / 1e9, 1),
            "host_issue_us_per_call": round(issue[0] * 1e6 / steps / len(wl.calls), 2),
            "method": ("activations only (weights, scales and biases resident, uploaded once "
                       "before the timed region); " if weights_resident else "") +
                      ("the 14 calls of a step replayed as one captured CUDA graph; "
                       if graphed else "") +
                      "packed pinned inputs copied in as two halves on two copy streams and "
                      "one packed D2H copy per step on a third; the next step's inputs move "
                      "in and the previous step's outputs move out while the current step "
                      "computes"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_steps(problems, min_seconds, max_steps=None, threads=None):
    """Run the oracle over the whole step (all 14 calls) until min_seconds
    have passed (at least one step); returns (seconds per step, steps)."""
    import oracle
    oracle.build()
    n, t0 = 0, time.perf_counter()
    while True:
        for p in problems:
            oracle.qmm(p["A"], p["Wq"], p["scales"], p["biases"], threads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or (max_steps and n >= max_steps):
            return el / n, n


def host_description():
    """The host the oracle ran on: machine, CPU model and logical CPUs."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if model is None:  # Arm hosts name the core in lscpu, not in /proc/cpuinfo
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name:"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"machine": platform.machine(), "cpu": model, "logical_cpus": os.cpu_count()}


def cpu_baseline(problems):
    import oracle
    threads = oracle.default_threads()
    sec, n = oracle_steps(problems, 10.0, threads=threads)
    # the small case (k projection at M = 16) on one thread, median of 3
    small = inputs.make_w4a16(16, *inputs.PROJECTIONS["k"], seed=0)
    one = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.qmm(small["A"], small["Wq"], small["scales"], small["biases"], threads=1)
        one.append(time.perf_counter() - t0)
    return {"value": round(sec * 1e6 / len(problems), 1), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": "%d full step(s) of the workload (all 14 calls, fp64 C = A.W^T) on %d "
                      "host threads" % (n, threads),
            "single_thread_small_us": round(statistics.median(one) * 1e6, 1),
            "single_thread_small": "k projection at M = 16 (Kred 2560, Nout 1024), one thread, "
                                   "median of 3",
            "host": host_description()}


def run_reference(args, rank, world):
    """The CPU oracle on the same workload.  Each step is a bounded sample:
    one call of the 14 (in turn), all M rows and a subset of the output
    columns sized so that warm-up and timed steps together take about 90 s;
    the sample's time is scaled to the whole call by Nout / columns (the
    oracle's cost is linear in the columns it computes)."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    problems = [inputs.make_w4a16(M, Kred, Nout, seed=0) for (_, M, Kred, Nout) in calls()]
    threads = oracle.default_threads()
    budget = max(0.02, 90.0 / (args.steps + args.warmup))
    rng = np.random.default_rng(0)

    def run(p, cols):
        rows = np.arange(p["M"])
        t0 = time.perf_counter()
        oracle.qmm_sampled(p["A"], p["Wq"], p["scales"], p["biases"], rows, cols, threads=threads)
        return time.perf_counter() - t0

    cols_of = []
    for p in problems:
        probe = np.arange(min(64, p["Nout"]))
        t = run(p, probe)
        nc = int(min(p["Nout"], max(8, len(probe) * budget / max(t, 1e-6))))
        cols_of.append(np.sort(rng.choice(p["Nout"], nc, replace=False)))
    for k in range(args.warmup):
        i = k % len(problems)
        run(problems[i], cols_of[i])
    est, wall = [], 0.0
    for k in range(args.steps):
        i = k % len(problems)
        t = run(problems[i], cols_of[i])
        wall += t
        est.append(t * problems[i]["Nout"] / len(cols_of[i]))
    value = round(statistics.mean(est) * 1e6, 1)
    sample = "each step: one of the 14 calls in turn, all M rows x %d..%d of Nout columns, " \
             "scaled to the full call by Nout/columns" % (min(len(c) for c in cols_of),
                                                          max(len(c) for c in cols_of))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall * 1e3 / max(1, args.steps), 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "calls_per_step": 1,
                       "oracle": "plain C, fp64 accumulate, OpenMP"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample, "host": host_description()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch-list", action="store_true",
                    help="only the timed graph steps (for a profiler's launch list)")
    ap.add_argument("--weights", choices=["static", "dynamic"], default="static",
                    help="static: promise that no kernel writes the weights during the run "
                         "(qmm_set_weights_static), which lets weight work start early")
    ap.add_argument("--kernels", choices=["default", "mma", "tc", "lean"], default="default",
                    help="kernel table for the W4A16 calls (A/B comparisons)")
    ap.add_argument("--partitions", choices=["equal", "near-equal"], default="equal",
                    help="partition rule of the W4A16 calls (qmm_set_partitions)")
    ap.add_argument("--only", default=None, metavar="PROJ:M",
                    help="restrict the step to one call, e.g. gate:128 (profiling aid)")
    ap.add_argument("--grouped", choices=["tiles", "persistent"], default=None,
                    help="with --launch-list: time the step's calls as one grouped call "
                         "under this schedule (profiling aid)")
    ap.add_argument("--group-plan", action="store_true",
                    help="with --grouped: splits planned for the group (qmm_set_group_plan)")
    ap.add_argument("--attention-only", action="store_true",
                    help="only the decode-attention calls at the plan's split (profiling aid)")
    ap.add_argument("--split-req", choices=["policy", "planned", "balanced"], default="policy",
                    help="with --launch-list: the split request of every call (profiling aid)")
    ap.add_argument("--dense-only", type=int, default=None, metavar="SPLIT",
                    help="only dense split-K GEMM calls at this split (profiling aid)")
    args = ap.parse_args()
    if args.only:
        global ONLY
        name, m = args.only.split(":")
        ONLY = (name, int(m))
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.grouped and not args.launch_list:
        ap.error("--grouped is a profiling aid of --launch-list")
    if args.group_plan and not args.grouped:
        ap.error("--group-plan applies to --grouped")
    if args.split_req != "policy" and not args.launch_list:
        ap.error("--split-req is a profiling aid of --launch-list")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.attention_only:
        return run_attention_only(args)
    if args.dense_only is not None:
        return run_dense_only(args)
    res = run_gpu(args, rank, world, local_rank)
    wl = res["wl"]
    ncalls = len(wl.calls)
    value_us = job_value_us(res["ms"], world, args.steps, ncalls)
    if res.get("launch_list"):
        if rank == 0:
            per_step = res["grouped_launches"] or wl.launches_per_step()
            print(json.dumps({"launch_list": True, "value": value_us, "unit": UNIT,
                              "steps": args.steps, "splits": res["splits"],
                              "grouped": args.grouped, "group_plan": args.group_plan,
                              "gpu_launches": args.steps * per_step}), flush=True)
        return

    dc = res["per_call"][res["dom"]["index"]]
    peaks = res["peaks"]
    from split_w4a16_quantized_gb300 import qmm as Q
    bm, bn = Q.qmm_kernel_tile(dc["M"])
    split = dc["split"]
    if split > 1:  # the partition kernel alone
        nb, fl = partition_algorithmic(dc["M"], dc["Kred"], dc["Nout"], split)
        us = res["dom"]["us_partition"]
        kernel = "partition kernel (%s), BM=%d BN=%d, grid %d x %d x %d" % (
            "tcgen05" if args.kernels != "mma" else "mma.sync", bm, bn,
            -(-dc["Nout"] // bn), -(-dc["M"] // bm), split)
    else:
        nb, fl = algorithmic(dc["M"], dc["Kred"], dc["Nout"], 1)
        us = dc["us_split"]
        kernel = "unsplit kernel, BM=%d BN=%d" % (bm, bn)
    _, bound = roofline_time_s(nb, fl, peaks)
    if bound == "hbm":
        achieved, peak, unit = nb / us / 1e3, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = fl / us / 1e6, peaks["bf16_tflops"], "TFLOP/s"
    traffic = None
    key = (dc["proj"], dc["M"], split)
    if args.kernels != "mma" and key in NCU_TRAFFIC and NCU_TRAFFIC[key][1] == tc_source_hash():
        traffic = NCU_TRAFFIC[key][0]
    roof = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "peak_source": res["peak_src"] + " (burst)", "kernel": kernel,
            "call": "%s M=%d Kred=%d Nout=%d split=%d" % (dc["proj"], dc["M"], dc["Kred"],
                                                        dc["Nout"], split),
            "per_launch": {"algorithmic_bytes": nb, "flops": fl, "us": round(us, 3)},
            "reduce_us": round(res["dom"].get("us_reduce", 0.0), 3),
            "timing": "CUDA events around replays of a graph of back-to-back launches of the "
                      "kernel alone, each launch on its own copy of the inputs (copies > 2.2x L2, "
                      "weights read from HBM); programmatic dependent launch on, no "
                      "static-weights early start"}
    roof_alt = None
    if "us_partition_alt" in res["dom"]:
        # the same kernel and call under the other partition rule
        s_alt = res["dom"]["split_alt"]
        nb_a, fl_a = partition_algorithmic(dc["M"], dc["Kred"], dc["Nout"], s_alt)
        us_a = res["dom"]["us_partition_alt"]
        ach_a = nb_a / us_a / 1e3 if bound == "hbm" else fl_a / us_a / 1e6
        key_a = (dc["proj"], dc["M"], s_alt)
        tr_a = NCU_TRAFFIC[key_a][0] if (args.kernels != "mma" and key_a in NCU_TRAFFIC and
                                         NCU_TRAFFIC[key_a][1] == tc_source_hash()) else None
        roof_alt = {"partitions": "near-equal" if args.partitions == "equal" else "equal",
                    "split": s_alt, "grid": "%d x %d x %d" % (-(-dc["Nout"] // bn),
                                                            -(-dc["M"] // bm), s_alt),
                    "achieved": round(ach_a, 2), "peak": peak, "unit": unit,
                    "frac": round(ach_a / peak, 4), "traffic": tr_a,
                    "per_launch": {"algorithmic_bytes": nb_a, "flops": fl_a, "us": round(us_a, 3)}}
    step_roof = step_roofline(wl, res["ms"] / args.steps, peaks)
    out = {"metric": METRIC, "value": round(value_us, 4), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(res["ms"] / args.steps, 6), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": WORKLOAD, "calls_per_step": ncalls,
                      "policy": policy_desc(),
                      "l2": "inputs larger than L2: %d rotating input sets x %.0f MB (L2 %d MB)"
                            % (wl.R, wl.set_bytes / 2**20, res["l2"] >> 20),
                      "kernels": args.kernels,
                      "partitions": "equal (the split divides the groups; the chapter's rule)"
                                    if args.partitions == "equal" else
                                    "near-equal (qmm_set_partitions: any split, the first "
                                    "G mod s partitions one group longer)",
                      "weights": "static (qmm_set_weights_static: no kernel writes the "
                                 "weights during the run; weight loads and dequant start "
                                 "before the previous kernel ends)" if args.weights == "static"
                                 else "dynamic (every kernel waits for the previous one)",
                      "graphs": "one CUDA graph per step, replayed", "parallelism":
                      "replicas x%d" % world, "sms": res["sms"]},
           "value_without_pdl": round(job_value_us(res["ms_nopdl"], 1, args.steps, ncalls), 4),
           ("value_weights_dynamic" if args.weights == "static" else "value_weights_static"):
               round(job_value_us(res["ms_wflip"], 1, args.steps, ncalls), 4),
           "value_fused_reduce": round(job_value_us(res["ms_fused"], 1, args.steps, ncalls), 4),
           "value_cluster_reduce": round(job_value_us(res["ms_cluster"], 1, args.steps, ncalls),
                                         4),
           ("value_near_equal" if args.partitions == "equal" else "value_equal_partitions"):
               round(job_value_us(res["ms_alt"], 1, args.steps, ncalls), 4),
           "value_grouped": round(job_value_us(res["ms_grouped"], 1, args.steps, ncalls), 4),
           "value_grouped_tiles": round(job_value_us(res["ms_grouped_tiles"], 1, args.steps,
                                                     ncalls), 4),
           "value_grouped_group_plan": round(job_value_us(res["ms_grouped_plan"], 1, args.steps,
                                                          ncalls), 4),
           "group_plan_splits": res["group_plan_splits"],
           "grouped_launches_per_step": res["grouped_launches"],
           "roofline": roof, "roofline_other_partitions": roof_alt, "step_roofline": step_roof,
           "gpu_launches": args.steps * wl.launches_per_step(),
           "clocks": res["clocks"], "e2e": res["e2e"],
           "e2e_weights_resident": res["e2e_resident"],
           "e2e_weights_resident_graphed": res["e2e_resident_graph"], "per_call": res["per_call"],
           "dense_splitk_512x512x16384": res["dense"], "prefill_M2048": res["prefill"],
           "split_vs_control": res["sweep"],
           "overlap_stream": res["overlap"], "decode_attention": res["attention"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl.host)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
