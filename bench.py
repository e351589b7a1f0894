#!/usr/bin/env python
"""Benchmark of the MMVQ hot path on GB300: weight GB/s per call at 1-8 columns.

Default workload: the Q6_K sweep -- 2560x2560, 2560x10240 and 10240x2560
(rows x K) at 1, 2, 4, 6 and 8 Q8_1 columns, weights repacked at load into
planar tiles -- the pages' mmvq_bench table ("Strata" PR #2207).  One step
is one pass over every (shape, columns) case on every resident copy of its
matrix; the copies of each shape total more than twice the L2 size, so no
call finds its weights in L2.  Per case the hot path runs as in decode: the
fp32 columns are quantised to Q8_1 once, then every matrix copy gets its
MMVQ call (several matrices sharing one activation, like q/k/v or gate/up).

The step's calls are made through the public binding and captured once as a
CUDA graph (the pages' figures are graph replays too, PR #2746).  `value` =
weight bytes of all calls / device time of that graph's replays.  Per-case
times come from a second capture of the same calls with event-record nodes at
the boundaries of each case, replayed after the timed region (an event node
ends the programmatic chaining of the launches around it, so it stays out of
the timed graph).  `e2e` repeats the step with the fp32 columns copied in
from pinned host memory, the calls made eagerly through the public binding
(the C ABI, one call at a time) and all outputs read back every step;
`e2e_graph` is the same with the calls replayed as the captured graph.

The default run also times the pages' other matrices (the LM head and the
gathered draft head at 1-5 columns, the Q4_K and Q5_K dense shapes, the MoE
layer at T = 1, 4, 8), each as its own workload with fewer steps, and
one-column decode steps as a dependent chain (quantiser + product against
the fused fp32 entry), and adds their summaries under `workloads`
(`--no-extra` leaves them out).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a row sample

Under torchrun each rank runs an independent replica (the path has no
exchange step); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

METRIC = "weight GB/s per MMVQ call (fraction of HBM peak) and us/call at 1-8 cols"
UNIT = "GB/s"

SWEEP_SHAPES = [(2560, 2560), (2560, 10240), (10240, 2560)]
SWEEP_COLS = [1, 2, 4, 6, 8]
HEAD_SHAPE = (151936, 2560)
DRAFT_ROWS = 4096
MOE = {"experts": 256, "hidden": 2560, "ffn": 768, "top_k": 8}
Q4K_SHAPES = [(12288, 2560), (6144, 2560), (2560, 6144), (640, 2560), (512, 2560)]


def workload_cases(name):
    """-> list of (fmt, rows, K, ncols_list)."""
    if name == "q6k_sweep":
        return [("q6_k_planar", r, k, SWEEP_COLS) for r, k in SWEEP_SHAPES]
    if name == "q6k_sweep_gguf":
        return [("q6_k", r, k, SWEEP_COLS) for r, k in SWEEP_SHAPES]
    if name == "lm_head":
        return [("q6_k_planar", HEAD_SHAPE[0], HEAD_SHAPE[1], [1, 2, 3, 4, 5]),
                ("q6_k_planar_draft", DRAFT_ROWS, HEAD_SHAPE[1], [1, 2, 3, 4, 5])]
    if name == "q4k_dense":
        return [("q4_k_planar", r, k, [1, 4]) for r, k in Q4K_SHAPES]
    if name == "q5k_dense":
        return [("q5_k_planar", r, k, [1, 4]) for r, k in Q4K_SHAPES]
    if name == "q4k_dense_gguf":
        return [("q4_k", r, k, [1, 4]) for r, k in Q4K_SHAPES]
    raise SystemExit(f"unknown workload {name}")


WORKLOAD_DESC = {
    "q6k_sweep": "Q6_K MMVQ sweep 2560x2560, 2560x10240, 10240x2560 (rows x K) at 1,2,4,6,8 cols, planar tiles",
    "q6k_sweep_gguf": "Q6_K MMVQ sweep 2560x2560, 2560x10240, 10240x2560 at 1,2,4,6,8 cols, GGUF blocks",
    "lm_head": "Q6_K LM head 151936x2560 at 1-5 cols, planar tiles; 4096-row draft head gathered from it",
    "q4k_dense": "Q4_K dense 12288x2560, 6144x2560, 2560x6144, 640x2560, 512x2560 at 1 and 4 cols, planar tiles",
    "q4k_dense_gguf": "Q4_K dense 12288x2560, 6144x2560, 2560x6144, 640x2560, 512x2560 at 1 and 4 cols, GGUF blocks",
    "q5k_dense": "Q5_K dense 12288x2560, 6144x2560, 2560x6144, 640x2560, 512x2560 at 1 and 4 cols, planar tiles",
    "moe_t1": "grouped MoE Q4_K, 256 experts, gate|up 1536x2560, down 2560x768, T=1 top-8 (planar experts)",
    "moe_t4": "grouped MoE Q4_K, 256 experts, gate|up 1536x2560, down 2560x768, T=4 top-8 (planar experts)",
    "moe_t8": "grouped MoE Q4_K, 256 experts, gate|up 1536x2560, down 2560x768, T=8 top-8 (planar experts)",
    "prologue": "RMSNorm folded into the Q8_1 quantiser vs the plain quantiser, K = 2560 and 10240 at 1, 4, 8 cols",
}


MMVQ_SOURCES = ["api.cu", "common.cuh", "expert_ffn.cu", "ffn_args.cuh", "kquant.cuh", "mmvq_dense.cu",
                "mmvq_tma.cu", "mmvq_tma_f32.cu", "q8_1.cuh", "ring.cuh", "route.cuh", "rowgroup.cuh",
                "tma_dense.cuh", "tma_mma.cuh"]


def kernel_source_hash() -> str:
    """sha256 of the sources the profiled kernels (dense ring, grouped ring,
    the one-launch expert layer, their launch choosers) are built from, and
    of the ABI header."""
    import hashlib
    h = hashlib.sha256()
    for p in [os.path.join(HERE, "block_quantized_matvec_gb300", "csrc", f) for f in MMVQ_SOURCES] + \
            [os.path.join(HERE, "include", "mmvq.h")]:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_field(summary: str, key: str):
    """A number from a committed ncu summary, or None when the summary is
    missing or was taken on different kernel sources."""
    try:
        text = open(os.path.join(HERE, "profiles", summary)).read()
    except OSError:
        return None
    fields = dict(l.split(": ", 1) for l in text.splitlines() if ": " in l and not l.startswith("|"))
    if fields.get("kernel_source_sha256", "").strip() != kernel_source_hash():
        return None
    try:
        return float(fields[key])
    except (KeyError, ValueError):
        return None


def profiled_traffic(summary: str):
    """DRAM bytes per MMVQ launch from a committed ncu summary (or None)."""
    v = profiled_field(summary, "traffic_bytes_per_mmvq_launch")
    return None if v is None else int(v)


def host_weights_for(fmt: str, rows: int, K: int, salt: int = 0):
    """Seeded GGUF blocks for a workload format (the planar forms repack them)."""
    from block_quantized_matvec_gb300 import synth
    gen = (synth.q4_k_weights if fmt.startswith("q4_k") else
           synth.q5_k_weights if fmt.startswith("q5_k") else synth.q6_k_weights)
    return gen(rows, K, salt=salt)


def repack_source(fmt: str) -> int:
    from block_quantized_matvec_gb300 import mmvq
    return (mmvq.TYPE_Q4_K if fmt.startswith("q4_k") else
            mmvq.TYPE_Q5_K if fmt.startswith("q5_k") else mmvq.TYPE_Q6_K)


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the slowest replica sets the job's
    time); the value itself with one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peak():
    p = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first_sample(self, timeout_s: float = 10.0):
        """nvidia-smi's start-up can stall the GPU: let it settle before timing."""
        t = time.time()
        while self.proc is not None and len(self.lines) < 2 and time.time() - t < timeout_s:
            time.sleep(0.02)

    def mark(self):
        self.first_timed = len(self.lines)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        timed = self.lines[getattr(self, "first_timed", 0):] or self.lines[-1:]
        for l in timed:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- graph events --

_cudart = None


def _record_external(ev, stream):
    """Event-record node inside a stream capture (cudaEventRecordExternal), so
    the event is timestamped every time the graph runs."""
    global _cudart
    if _cudart is None:
        _cudart = ctypes.CDLL("libcudart.so.13")
        _cudart.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        _cudart.cudaEventRecordWithFlags.restype = ctypes.c_int
    rc = _cudart.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event),
                                          ctypes.c_void_p(stream.cuda_stream), 1)
    if rc != 0:
        raise RuntimeError(f"cudaEventRecordWithFlags failed ({rc})")


# -------------------------------------------------------------- our arm --

def run_ours(args, rank, world, local_rank):
    import torch
    from block_quantized_matvec_gb300 import metrics, mmvq, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    mmvq.lib()

    cases_spec = workload_cases(args.workload)
    type_of = {"q6_k_planar": mmvq.TYPE_Q6_K_PLANAR, "q6_k": mmvq.TYPE_Q6_K, "q4_k": mmvq.TYPE_Q4_K,
               "q4_k_planar": mmvq.TYPE_Q4_K_PLANAR, "q6_k_planar_draft": mmvq.TYPE_Q6_K_PLANAR,
               "q5_k_planar": mmvq.TYPE_Q5_K_PLANAR}

    # resident weights: copies per shape so that each shape's copies exceed 2x L2
    mats = []
    host_weights = []
    for si, (fmt, rows, K, cols) in enumerate(cases_spec):
        if fmt == "q6_k_planar_draft":
            # the draft head: seeded rows gathered from the planar LM head above
            head_rows = cases_spec[0][1]
            ids = synth.draft_rows(rows, head_rows)
            Wd, _ = mmvq.gather_planar_rows(mats[0][0], head_rows, K,
                                            torch.from_numpy(ids).to(dev))
            host_weights.append(np.ascontiguousarray(host_weights[0][ids]))
        else:
            W = host_weights_for(fmt, rows, K, salt=si)
            host_weights.append(W)
            Wd = torch.from_numpy(W.reshape(-1)).to(dev)
            if fmt.endswith("_planar"):
                Wd = mmvq.repack_planar(Wd, rows, K, type_=repack_source(fmt))
        nbytes = metrics.weight_bytes(fmt, rows, K)
        copies = max(2, math.ceil(2 * l2 / nbytes))
        mats.append([Wd] + [Wd.clone() for _ in range(copies - 1)])
    torch.cuda.synchronize()

    # activations of every (shape, ncols) case, in one buffer (one H2D per step for e2e)
    case_list = []
    x_total = 0
    for si, (fmt, rows, K, cols) in enumerate(cases_spec):
        for nc in cols:
            case_list.append((si, fmt, rows, K, nc, x_total))
            x_total += nc * K
    x_host = np.concatenate([synth.activations(K, nc, salt=100 * si + nc).reshape(-1)
                             for (si, fmt, rows, K, nc, _) in case_list])
    x_dev = torch.from_numpy(x_host).to(dev)
    x_pinned = torch.from_numpy(x_host).pin_memory()
    xq_bufs = [torch.empty((nc, K // 32, 36), dtype=torch.uint8, device=dev)
               for (_, _, _, K, nc, _) in case_list]

    calls = []  # (case index, copy index, y offset)
    y_total = 0
    for ci, (si, fmt, rows, K, nc, xo) in enumerate(case_list):
        for cp in range(len(mats[si])):
            calls.append((ci, cp, y_total))
            y_total += nc * rows
    y_dev = torch.empty(y_total, dtype=torch.float32, device=dev)
    y_pinned = torch.empty(y_total, dtype=torch.float32).pin_memory()
    calls_of_case = [[i for i, c in enumerate(calls) if c[0] == ci] for ci in range(len(case_list))]

    # the views each call takes, made once (as a caller with preallocated
    # buffers would)
    x_views = [x_dev[xo:xo + nc * K].view(nc, K) for (_, _, _, K, nc, xo) in case_list]
    y_views = [y_dev[yo:yo + case_list[ci][4] * case_list[ci][2]].view(case_list[ci][4],
                                                                       case_list[ci][2])
               for (ci, _, yo) in calls]

    def run_case(ci, s=None, evs=None, dependent=False):
        """Quantise the case's columns once, then every copy's MMVQ back to back.
        dependent=True drops the stable-activation flag: every call then waits
        for its predecessor before it stages the activations (a chain of
        calls that each consume the previous result)."""
        si, fmt, rows, K, nc, xo = case_list[ci]
        if evs is not None:
            _record_external(evs[3 * ci], s)
        mmvq.quantize_q8_1(x_views[ci], out=xq_bufs[ci])
        if evs is not None:
            _record_external(evs[3 * ci + 1], s)
        t = type_of[fmt]
        for n, i in enumerate(calls_of_case[ci]):
            # after the first call no kernel that may still run writes xq
            mmvq.gemv(t, mats[si][calls[i][1]], rows, K, xq_bufs[ci], nc, out=y_views[i],
                      flags=mmvq.FLAG_XQ_STABLE if (n and not dependent) else 0)
        if evs is not None:
            _record_external(evs[3 * ci + 2], s)

    # first calls outside any capture (kernel attributes, launch shapes)
    for ci in range(len(case_list)):
        run_case(ci)
    torch.cuda.synchronize()

    # the step as one CUDA graph, every launch chained to the previous one by
    # programmatic dependent launch; a second capture of the same calls with
    # event nodes at the case boundaries gives the per-case times
    def capture(evs=None, dependent=False):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            s = torch.cuda.current_stream()
            for ci in range(len(case_list)):
                run_case(ci, s, evs, dependent)
        torch.cuda.synchronize()
        return g

    def events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3 * len(case_list))]
        for e in evs:
            e.record()
        torch.cuda.synchronize()
        return evs

    cap = torch.cuda.Stream(device=dev)
    graph = capture()
    evs = events()
    graph_ev = capture(evs)

    stream = torch.cuda.current_stream()
    import torch.distributed as dist
    gpu_index = local_rank
    if "CUDA_VISIBLE_DEVICES" in os.environ:
        vis = os.environ["CUDA_VISIBLE_DEVICES"].split(",")
        if local_rank < len(vis) and vis[local_rank].strip().isdigit():
            gpu_index = int(vis[local_rank])
    clocks = ClockSampler(gpu_index)
    clocks.start()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks.wait_first_sample()
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks.mark()
    t0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    barrier(world)

    def case_times(g, ev, runs=5):
        """Median over replays of (quantise, MMVQ calls) time per case, in us."""
        for _ in range(2):
            g.replay()
        samples = []
        for _ in range(runs):
            g.replay()
            torch.cuda.synchronize()
            samples.append([[ev[3 * ci + j].elapsed_time(ev[3 * ci + j + 1]) * 1e3 for j in (0, 1)]
                            for ci in range(len(case_list))])
        med = np.median(np.array(samples), axis=0)
        return med[:, 0], med[:, 1]

    # per-case durations from the instrumented capture (outside the timed region)
    q_us, g_us = case_times(graph_ev, evs)
    # the same calls as a dependent chain: each waits for its predecessor
    evd = events()
    _, d_us = case_times(capture(evd, dependent=True), evd)

    peak, peak_kind = load_peak()
    w_step = 0
    alg_step = 0
    per_case = []
    for ci, (si, fmt, rows, K, nc, xo) in enumerate(case_list):
        n = len(calls_of_case[ci])
        wb = metrics.weight_bytes(fmt, rows, K)
        w_step += wb * n
        alg_step += metrics.call_bytes(fmt, rows, K, nc) * n
        gu = float(g_us[ci]) / n
        du = float(d_us[ci]) / n
        per_case.append({"shape": f"{rows}x{K}", "fmt": fmt, "ncols": nc, "calls": n,
                         "launch": mmvq.launch_shape(type_of[fmt], rows, K, nc),
                         "us_per_call": round(gu, 3), "us_quantize": round(float(q_us[ci]), 3),
                         "weight_gbps": round(wb / gu / 1e3, 1),
                         "frac_of_measured": round(wb / gu / 1e3 / peak, 3),
                         "us_per_call_dependent": round(du, 3),
                         "weight_gbps_dependent": round(wb / du / 1e3, 1)})
    step_s = elapsed_ms / 1e3 / args.steps
    value = world * w_step / step_s / 1e9
    # the MMVQ launches' algorithmic bytes over the timed step (which also
    # holds one Q8_1 launch per case: a conservative figure)
    achieved = alg_step / step_s / 1e9
    achieved_instr = alg_step / (float(np.sum(g_us)) * 1e-6) / 1e9

    # e2e: every step, H2D of the step's fp32 columns from pinned memory, the
    # step's calls made eagerly through the public binding (each a ctypes call
    # into the C ABI: argument checks, launch), D2H of every output, a
    # synchronise; the same with the calls replayed as the captured graph is
    # reported beside it (e2e_graph).  Left out for the extra workloads.
    e2e_steps = 0 if getattr(args, "light", False) else max(3, min(args.steps // 3, 100))

    def e2e_time(replay):
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for _ in range(e2e_steps):
            x_dev.copy_(x_pinned, non_blocking=True)
            if replay:
                graph.replay()
            else:
                for ci in range(len(case_list)):
                    run_case(ci)
            y_pinned.copy_(y_dev, non_blocking=True)
            torch.cuda.synchronize()
        return max_over_ranks((time.perf_counter() - w0) / max(1, e2e_steps), world, dev)

    e2e_s = e2e_time(False) if e2e_steps else 1.0
    e2e_graph_s = e2e_time(True) if e2e_steps else 1.0

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 dp4a + fp32",
        "data": "synthetic (seeded generators shaped like the pages' matrices)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "calls_per_step": len(calls),
                   "weight_copies": [len(m) for m in mats],
                   "l2": "weights rotated over copies > 2x L2 per shape (inputs larger than L2)",
                   "timing": "CUDA graph replay of the step (no event nodes inside); per-case "
                             "times: median of 5 replays of the same calls captured with event "
                             "nodes at case boundaries, after the timed region",
                   "instrumented_step_ms": round(float(np.sum(q_us) + np.sum(g_us)) / 1e3, 4),
                   "chain": "calls after a case's first carry the stable-activation flag, so "
                            "consecutive calls overlap; *_dependent per case: the same calls "
                            "without it (each waits for its predecessor), timed after the step",
                   "step": "per case: Q8_1-quantise its columns once, then one MMVQ per weight copy",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3),
                     "traffic": (profiled_traffic("mmvq_q6k_sweep_launch_list.md")
                                 if args.workload == "q6k_sweep" else None),
                     "algorithmic_bytes_per_launch": round(alg_step / len(calls)),
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "kernel": "MMVQ kernel, all launches of the timed step (its one Q8_1 launch "
                               "per case counted in the time)",
                     "achieved_instrumented": round(achieved_instr, 1)},
        "e2e": ({"value": round(world * w_step / e2e_s / 1e9, 1), "unit": UNIT,
                 "h2d_bytes_per_step": int(x_host.nbytes), "d2h_bytes_per_step": int(y_total * 4),
                 "steps": e2e_steps, "ms_per_step": round(e2e_s * 1e3, 3),
                 "calls": "eager: mmvq.quantize_q8_1 + mmvq.gemv per case through the C ABI"}
                if e2e_steps else None),
        "e2e_graph": ({"value": round(world * w_step / e2e_graph_s / 1e9, 1), "unit": UNIT,
                       "ms_per_step": round(e2e_graph_s * 1e3, 3),
                       "calls": "the same calls replayed as the captured CUDA graph"}
                      if e2e_steps else None),
        "gpu_launches": (len(calls) + len(case_list)) * args.steps,
        "clocks": clk,
        "cases": per_case,
        "dependent_chain": {"weight_gbps": round(w_step / (float(np.sum(d_us)) * 1e-6) / 1e9, 1),
                            "mmvq_us_per_step": round(float(np.sum(d_us)), 1),
                            "note": "MMVQ launches only, each call waiting for the previous"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cases_spec, host_weights, args.cpu_seconds)
    return out



# ------------------------------------------------------------- MoE step --

def run_moe(args, rank, world, local_rank):
    """One step = the routed-expert FFN of one MoE layer for T tokens in one
    launch (mmvq_expert_ffn): the per-expert token lists from the top-k
    routing, Q8_1 of the hidden states, grouped gate|up MMVQ, SiLU(gate)*up
    requantised to Q8_1, grouped down MMVQ.  The same step as the four
    separate launches (quantise + route, grouped gate|up, SiLU*up -> Q8_1,
    grouped down) is timed beside it as `chain`.
    Experts are planar Q4_K tiles; step i uses routing i mod 16, so
    consecutive steps read different experts (the 16 routings together touch
    far more expert bytes than L2 holds).  Each timed region is one CUDA graph
    of exactly K steps.  Weight bytes = distinct experts read x (gate|up +
    down) bytes."""
    import torch
    from block_quantized_matvec_gb300 import metrics, mmvq, synth

    T = int(args.workload.split("_t")[1])
    E, H, F, k = MOE["experts"], MOE["hidden"], MOE["ffn"], MOE["top_k"]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mmvq.lib()
    q4 = mmvq.TYPE_Q4_K

    def planar_experts(rows, K, salt):
        host = synth.expert_weights("q4_k", E, rows, K, salt=salt)
        per = mmvq.planar_bytes(rows, K, q4)
        out = torch.empty(E * per, dtype=torch.uint8, device=dev)
        for e in range(E):
            mmvq.repack_planar(torch.from_numpy(host[e].reshape(-1)).to(dev), rows, K,
                               out=out[e * per:(e + 1) * per], type_=q4)
        return out

    W_gu = planar_experts(2 * F, H, 1)
    W_dn = planar_experts(H, F, 2)
    R = 16
    topks = [synth.routing(T, k, E, salt=100 + r) for r in range(R)]
    topk_dev = [torch.from_numpy(t).to(dev) for t in topks]
    x_host = synth.moe_hidden(H, T)
    x_dev = torch.from_numpy(x_host).to(dev)
    x_pinned = torch.from_numpy(x_host).pin_memory()
    topk_pinned = torch.from_numpy(topks[0]).pin_memory()
    topk_e2e = torch.empty_like(topk_dev[0])
    n = T * k
    xq = torch.empty((T, H // 32, 36), dtype=torch.uint8, device=dev)
    gu = torch.empty((n, 2 * F), device=dev)
    hq = torch.empty((n, F // 32, 36), dtype=torch.uint8, device=dev)
    y = torch.empty((n, H), device=dev)
    y_pinned = torch.empty((n, H)).pin_memory()
    lists = dict(expert_ids=torch.empty(E, dtype=torch.int32, device=dev),
                 offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                 act_index=torch.empty(n, dtype=torch.int32, device=dev),
                 slot_of=torch.empty(n, dtype=torch.int32, device=dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sync = mmvq.expert_ffn_workspace(dev)

    def fused(topk):
        # the layer in one launch (token lists written for a later combine)
        mmvq.lib().mmvq_expert_ffn(
            mmvq.TYPE_Q4_K_PLANAR, W_gu.data_ptr(), W_dn.data_ptr(), E, H, F, x_dev.data_ptr(), H,
            T, topk.data_ptr(), k, gu.data_ptr(), hq.data_ptr(), y.data_ptr(),
            lists["expert_ids"].data_ptr(), lists["offsets"].data_ptr(),
            lists["act_index"].data_ptr(), lists["slot_of"].data_ptr(), xq.data_ptr(),
            status.data_ptr(), sync.data_ptr(), torch.cuda.current_stream().cuda_stream)

    def chain(topk, evs=None, s=None):
        rec = (lambda i: _record_external(evs[i], s)) if evs is not None else (lambda i: None)
        rec(0)
        _, eids, offs, act, _, st = mmvq.quantize_route_groups(x_dev, topk, E, xq=xq)
        rec(1)
        mmvq.grouped(mmvq.TYPE_Q4_K_PLANAR, W_gu, E, 2 * F, H, eids, offs, act, xq, T, n, out=gu,
                     status=st)
        rec(2)
        mmvq.silu_mul_quantize_q8_1(gu, F, out=hq)
        rec(3)
        mmvq.grouped(mmvq.TYPE_Q4_K_PLANAR, W_dn, E, H, F, eids, offs, None, hq, n, n, out=y,
                     status=st)
        rec(4)

    def capture(fn, n_steps, first=0):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            for i in range(n_steps):
                fn(topk_dev[(first + i) % R])
        torch.cuda.synchronize()
        return g

    for r in range(R):
        fused(topk_dev[r])
        chain(topk_dev[r])
    torch.cuda.synchronize()
    if int(status.item()) != 0 or mmvq.read_device_fault() != 0:
        raise RuntimeError("expert FFN reported a routing error or a device fault")
    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first_sample()
    timed = {}
    stream = torch.cuda.current_stream()
    for name, fn in (("fused", fused), ("chain", chain)):
        warm = capture(fn, max(3, args.warmup), first=R - 1)
        g = capture(fn, args.steps)
        warm.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        if name == "fused":
            clocks.mark()
        t0.record(stream)
        g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        timed[name] = max_over_ranks(t0.elapsed_time(t1), world, dev)
        barrier(world)
        del g, warm
    clk = clocks.stop()

    # the chain's kernels one by one: a graph per routing with event nodes
    # between the four launches, replayed after the timed regions
    dur_runs = []
    for r in range(R):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in evs:
            e.record()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            chain(topk_dev[r], evs, torch.cuda.current_stream())
        torch.cuda.synchronize()
        for rep in range(4):
            g.replay()
            torch.cuda.synchronize()
            dur_runs.append([evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(4)])

    distinct = [len(np.unique(t)) for t in topks]
    step_bytes = [metrics.moe_step_bytes(d, H, F) for d in distinct]
    total_bytes = sum(step_bytes[i % R] for i in range(args.steps))
    names = ["quantize_and_route", "grouped_gate_up", "silu_requant", "grouped_down"]
    mean_us = np.array(dur_runs).mean(axis=0)
    gu_bytes = np.mean([d * metrics.weight_bytes("q4_k", 2 * F, H) for d in distinct])
    dn_bytes = np.mean([d * metrics.weight_bytes("q4_k", H, F) for d in distinct])
    peak, peak_kind = load_peak()
    fused_ms = timed["fused"]
    # the fused kernel is the whole step: its algorithmic bytes per launch are
    # the step's weight bytes plus the activations it reads and writes
    act_bytes = T * H * 4 + T * (H // 32) * 36 + n * (2 * F * 4 * 2 + (F // 32) * 36 * 2 + H * 4)
    launch_bytes = float(np.mean(step_bytes)) + act_bytes
    achieved = launch_bytes / (fused_ms * 1e-3 / args.steps) / 1e9
    # DRAM bytes per launch: the profiled traffic / weight-byte ratio (T=8
    # capture) applied to this run's mean weight bytes
    ratio = profiled_field("mmvq_expert_ffn_moe_t1_t8.md", "traffic_over_weight_bytes")
    traffic = None if ratio is None else round(ratio * float(np.mean(step_bytes)))

    e2e_steps = 0 if getattr(args, "light", False) else max(3, min(args.steps, 200))
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for i in range(e2e_steps):
        x_dev.copy_(x_pinned, non_blocking=True)
        topk_e2e.copy_(topk_pinned, non_blocking=True)
        mmvq.expert_ffn(mmvq.TYPE_Q4_K_PLANAR, W_gu, W_dn, E, H, F, x_dev, topk_e2e, gu=gu, hq=hq,
                        y=y, xq=xq, sync=sync, lists=False)
        y_pinned.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - w0) / max(1, e2e_steps), world, dev)
    if mmvq.read_device_fault() != 0:
        raise RuntimeError("device fault word set after the timed runs")
    e2e_bytes = metrics.moe_step_bytes(distinct[0], H, F)

    out = {
        "metric": METRIC, "value": round(world * total_bytes / (fused_ms * 1e-3) / 1e9, 1),
        "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(fused_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 dp4a + fp32",
        "data": "synthetic (seeded generators shaped like the pages' matrices)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "tokens": T, "routings": R,
                   "parallelism": f"replicas x{world}",
                   "distinct_experts_mean": float(np.mean(distinct)),
                   "l2": "inputs larger than L2: 16 routings cycled, their experts far exceed L2",
                   "timing": "one CUDA graph of exactly `steps` steps per path"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3), "traffic": traffic,
                     "algorithmic_bytes_per_launch": round(launch_bytes),
                     "peak_kind": f"{peak_kind} hbm_gbs", "kernel": "mmvq_expert_ffn_kernel"},
        "e2e": ({"value": round(world * e2e_bytes / e2e_s / 1e9, 1), "unit": UNIT,
                 "h2d_bytes_per_step": int(x_host.nbytes + topks[0].nbytes),
                 "d2h_bytes_per_step": int(y.numel() * 4), "steps": e2e_steps,
                 "call": "mmvq.expert_ffn, routing 0 every step"} if e2e_steps else None),
        "gpu_launches": args.steps,
        "clocks": clk,
        "chain": {"ms_per_step": round(timed["chain"] / args.steps, 4),
                  "value": round(world * total_bytes / (timed["chain"] * 1e-3) / 1e9, 1),
                  "launches_per_step": 4,
                  "kernels_us": {nm: round(float(v), 3) for nm, v in zip(names, mean_us)},
                  "grouped_gbps": {"gate_up": round(gu_bytes / mean_us[1] / 1e3, 1),
                                   "down": round(dn_bytes / mean_us[3] / 1e3, 1)},
                  "note": "kernels_us from a graph with event nodes between the launches"},
    }
    return out

# ------------------------------------------------ activation prologue --

def run_prologue(args, rank, world, local_rank):
    """Per call: RMSNorm + Q8_1 of ncols columns (x and w read, Q8_1 written)
    against the plain Q8_1 quantiser of the same columns; CUDA graphs of
    back-to-back calls, inputs L2-resident (they are a few hundred KB)."""
    import torch
    from block_quantized_matvec_gb300 import mmvq, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    mmvq.lib()
    n_calls = 200
    cases = []
    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first_sample()
    clocks.mark()
    total_bytes, total_s = 0.0, 0.0
    for K in (2560, 10240):
        w = torch.from_numpy(synth.activations(K, 1, salt=K)[0]).to(dev)
        for nc in (1, 4, 8):
            x = torch.from_numpy(synth.activations(K, nc, salt=K + nc)).to(dev)
            xq = torch.empty((nc, K // 32, 36), dtype=torch.uint8, device=dev)
            row = {"K": K, "ncols": nc}
            for name, fn in (("rmsnorm_q8_1", lambda: mmvq.rmsnorm_quantize_q8_1(x, w, 1e-6, out=xq)),
                             ("q8_1", lambda: mmvq.quantize_q8_1(x, out=xq))):
                fn()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream(device=dev)
                cap.wait_stream(torch.cuda.current_stream())
                with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                    for _ in range(n_calls):
                        fn()
                for _ in range(max(3, args.warmup)):
                    g.replay()
                torch.cuda.synchronize()
                reps = 5
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                t0.record()
                for _ in range(reps):
                    g.replay()
                t1.record()
                torch.cuda.synchronize()
                us = t0.elapsed_time(t1) * 1e3 / (reps * n_calls)
                row[f"us_{name}"] = round(us, 3)
                if name == "rmsnorm_q8_1":
                    nbytes = 4 * K * nc + 4 * K + 36 * (K // 32) * nc
                    total_bytes += nbytes * reps * n_calls
                    total_s += us * 1e-6 * reps * n_calls
            cases.append(row)
    clk = clocks.stop()
    return {
        "metric": "RMSNorm+Q8_1 prologue: bytes moved (x, w in; Q8_1 out) per second",
        "value": round(total_bytes / total_s / 1e9, 2), "unit": "GB/s", "n_gpus": world,
        "steps": n_calls, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp64 mean square + fp32",
        "data": "synthetic N(0,1) columns and weights",
        "config": {"workload": WORKLOAD_DESC["prologue"], "eps": 1e-6,
                   "timing": "CUDA graph of 200 back-to-back calls, 5 replays"},
        "gpu_launches": len(cases) * 2 * n_calls * 5, "clocks": clk, "cases": cases,
    }


# ---------------------------------------------------------- CPU oracle --

def _oracle_pass(cases_spec, host_weights, row_sample, salt0=0):
    """One pass of the oracle over every case; returns (weight bytes, seconds)."""
    import oracle
    from block_quantized_matvec_gb300 import metrics, synth
    tcode = {"q6_k_planar": oracle.TYPE_Q6_K, "q6_k": oracle.TYPE_Q6_K, "q4_k": oracle.TYPE_Q4_K,
             "q4_k_planar": oracle.TYPE_Q4_K, "q6_k_planar_draft": oracle.TYPE_Q6_K,
             "q5_k_planar": oracle.TYPE_Q5_K}
    nbytes = 0
    secs = 0.0
    for si, (fmt, rows, K, cols) in enumerate(cases_spec):
        W = host_weights[si]
        r = rows if row_sample is None else min(rows, row_sample)
        Ws = W if r == rows else np.ascontiguousarray(W[:r])
        for nc in cols:
            x = synth.activations(K, nc, salt=100 * si + nc)
            t = time.perf_counter()
            xq = oracle.quantize_q8_1(x)
            oracle.gemv(tcode[fmt], Ws, r, K, xq, nc)
            secs += time.perf_counter() - t
            nbytes += metrics.weight_bytes(fmt, r, K)
    return nbytes, secs


def cpu_baseline(cases_spec, host_weights, seconds):
    import oracle
    oracle.build()
    nb_total, s_total, passes = 0, 0.0, 0
    while passes < 1 or (s_total < seconds and passes < 50):
        nb, s = _oracle_pass(cases_spec, host_weights, None)
        nb_total += nb
        s_total += s
        passes += 1
    return {"value": round(nb_total / s_total / 1e9, 3), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"{passes} full pass(es) of every case (all rows, all columns), "
                      f"{s_total:.1f} s single-threaded on {os.cpu_count()} host cores"}


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, each step a row sample of every case."""
    if rank != 0:
        return None
    from block_quantized_matvec_gb300 import synth
    import oracle
    oracle.build()
    cases_spec = workload_cases(args.workload)
    sample_rows = 64
    host_weights = []
    for si, (fmt, rows, K, cols) in enumerate(cases_spec):
        host_weights.append(np.ascontiguousarray(host_weights_for(fmt, min(rows, sample_rows), K,
                                                                  salt=si)))
    for _ in range(args.warmup):
        _oracle_pass(cases_spec, host_weights, sample_rows)
    nb_total, s_total = 0, 0.0
    for _ in range(args.steps):
        nb, s = _oracle_pass(cases_spec, host_weights, sample_rows)
        nb_total += nb
        s_total += s
    v = nb_total / s_total / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(s_total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32 + fp32 (oracle)",
        "data": "synthetic (seeded generators shaped like the pages' matrices)",
        "config": {"workload": WORKLOAD_DESC[args.workload], "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {sample_rows} rows of every case per step, all columns"},
        "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------ one-column decode steps --

DECODE_SHAPES = [("q6_k_planar", 2560, 2560), ("q6_k_planar", 2560, 10240),
                 ("q6_k_planar", 10240, 2560), ("q4_k_planar", 12288, 2560),
                 ("q6_k_planar", HEAD_SHAPE[0], HEAD_SHAPE[1])]


def run_decode(args, rank, world, local_rank):
    """One decode step per matrix: an fp32 column in, y out, each step waiting
    for the previous one (a dependent chain over rotating weight copies > 2x
    L2).  Two ways, timed as CUDA graphs of the same steps: the quantiser and
    the product as two launches (mmvq_quantize_q8_1, mmvq_gemv), and
    mmvq_gemv_f32 (one launch where the CTAs quantise the column themselves).
    us per step and weight GB/s for each."""
    import torch
    from block_quantized_matvec_gb300 import metrics, mmvq, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    type_of = {"q6_k_planar": mmvq.TYPE_Q6_K_PLANAR, "q4_k_planar": mmvq.TYPE_Q4_K_PLANAR}
    peak, _ = load_peak()
    cases = []
    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first_sample()
    clocks.mark()
    for si, (fmt, rows, K) in enumerate(DECODE_SHAPES):
        t = type_of[fmt]
        W = torch.from_numpy(host_weights_for(fmt, rows, K, salt=si).reshape(-1)).to(dev)
        W = mmvq.repack_planar(W, rows, K, type_=repack_source(fmt))
        wb = metrics.weight_bytes(fmt, rows, K)
        copies = max(2, math.ceil(2 * l2 / wb))
        mats = [W] + [W.clone() for _ in range(copies - 1)]
        x = torch.from_numpy(synth.activations(K, 1, salt=50 + si)).to(dev)
        xq = torch.empty((1, K // 32, 36), dtype=torch.uint8, device=dev)
        y = torch.empty((1, rows), device=dev)
        n = max(copies, 20 if wb > 1e8 else 100)

        def two(i):
            mmvq.quantize_q8_1(x, out=xq)
            mmvq.gemv(t, mats[i % copies], rows, K, xq, 1, out=y)

        def one(i):
            mmvq.gemv_f32(t, mats[i % copies], rows, K, x, 1, xq=xq, out=y)

        res = {}
        for name, fn in (("quantize_then_gemv", two), ("gemv_f32", one)):
            for i in range(copies):
                fn(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(device=dev)
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                for i in range(n):
                    fn(i)
            torch.cuda.synchronize()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            best = 1e30
            for _ in range(5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                best = min(best, e0.elapsed_time(e1) * 1e3 / n)
            us = max_over_ranks(best, world, dev)
            res[name] = {"us_per_step": round(us, 3), "weight_gbps": round(wb / us / 1e3, 1),
                         "frac_of_measured": round(wb / us / 1e3 / peak, 3)}
            del g
        cases.append({"shape": f"{rows}x{K}", "fmt": fmt,
                      "one_launch": mmvq.gemv_f32_fused(t, rows, K, 1), **res})
        del mats
        torch.cuda.empty_cache()
    return {"workload": "one-column decode steps as a dependent chain: the quantiser and the "
                        "product as two launches against mmvq_gemv_f32",
            "cases": cases, "clocks": clocks.stop()}


TENSOR_CORE_SHAPES = [("q6_k_planar", 2560, 2560), ("q6_k_planar", 2560, 10240),
                      ("q6_k_planar", 10240, 2560), ("q4_k_planar", 12288, 2560)]


def run_tensor_core(args, rank, world, local_rank):
    """The tensor-core consumer (MMVQ_FLAG_TENSOR_CORE) against the default
    dp4a consumer in the same launch shape, at 4, 6 and 8 columns: calls
    back to back (each after the first with MMVQ_FLAG_XQ_STABLE) over
    rotating weight copies > 2x L2, as CUDA graphs; us per call for each and
    whether y has the same bits."""
    import torch
    from block_quantized_matvec_gb300 import metrics, mmvq, synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20))
    type_of = {"q6_k_planar": mmvq.TYPE_Q6_K_PLANAR, "q4_k_planar": mmvq.TYPE_Q4_K_PLANAR}
    cases = []
    clocks = ClockSampler(local_rank)
    clocks.start()
    clocks.wait_first_sample()
    clocks.mark()
    for si, (fmt, rows, K) in enumerate(TENSOR_CORE_SHAPES):
        t = type_of[fmt]
        W = torch.from_numpy(host_weights_for(fmt, rows, K, salt=si).reshape(-1)).to(dev)
        W = mmvq.repack_planar(W, rows, K, type_=repack_source(fmt))
        wb = metrics.weight_bytes(fmt, rows, K)
        copies = max(2, math.ceil(2 * l2 / wb))
        mats = [W] + [W.clone() for _ in range(copies - 1)]
        n = max(copies, 100)
        for nc in (4, 6, 8):
            xq = mmvq.quantize_q8_1(torch.from_numpy(synth.activations(K, nc, salt=70 + si)).to(dev))
            y = torch.empty((nc, rows), device=dev)
            res = {}
            for name, base in (("dp4a", 0), ("tensor_core", mmvq.FLAG_TENSOR_CORE)):
                def fn(i, base=base):
                    mmvq.gemv(t, mats[i % copies], rows, K, xq, nc, out=y,
                              flags=base | (mmvq.FLAG_XQ_STABLE if i else 0))
                for i in range(copies):
                    fn(i)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                cap = torch.cuda.Stream(device=dev)
                cap.wait_stream(torch.cuda.current_stream())
                with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                    for i in range(n):
                        fn(i)
                torch.cuda.synchronize()
                for _ in range(3):
                    g.replay()
                torch.cuda.synchronize()
                best = 1e30
                for _ in range(5):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                    g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    best = min(best, e0.elapsed_time(e1) * 1e3 / n)
                res[name] = round(max_over_ranks(best, world, dev), 3)
                del g
            y0 = mmvq.gemv(t, mats[0], rows, K, xq, nc)
            y1 = mmvq.gemv(t, mats[0], rows, K, xq, nc, flags=mmvq.FLAG_TENSOR_CORE)
            cases.append({"shape": f"{rows}x{K}", "fmt": fmt, "ncols": nc,
                          "us_per_call_dp4a": res["dp4a"],
                          "us_per_call_tensor_core": res["tensor_core"],
                          "same_bits": bool(torch.equal(y0.view(torch.int32), y1.view(torch.int32)))})
        del mats
        torch.cuda.empty_cache()
    return {"workload": "4-8 columns, the tensor-core consumer (MMVQ_FLAG_TENSOR_CORE) against the "
                        "dp4a consumer in the same launch shape, calls back to back",
            "cases": cases, "clocks": clocks.stop()}


# --------------------------------------- the other workloads, summarised --

EXTRA_WORKLOADS = ["lm_head", "q4k_dense", "q5k_dense", "moe_t1", "moe_t4", "moe_t8"]


def run_extras(args, rank, world, local_rank):
    """The pages' other matrices, each timed as its own workload (fewer steps,
    no e2e or CPU leg) and summarised beside the sweep's line: per case
    us/call chained and dependent, weight GB/s and fraction of measured HBM;
    per MoE step us/layer for the one-launch layer and the four launches."""
    import gc

    import torch
    out = {}
    for w in EXTRA_WORKLOADS:
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup = w, args.extra_steps, 3
        sub.no_cpu_baseline, sub.light = True, True
        if w.startswith("moe_"):
            r = run_moe(sub, rank, world, local_rank)
            out[w] = {"workload": WORKLOAD_DESC[w], "us_per_layer": round(r["ms_per_step"] * 1e3, 2),
                      "weight_gbps": r["value"], "roofline_frac": r["roofline"]["frac"],
                      "distinct_experts_mean": r["config"]["distinct_experts_mean"],
                      "four_launches_us_per_layer": round(r["chain"]["ms_per_step"] * 1e3, 2),
                      "steps": sub.steps, "clocks": r["clocks"]}
        else:
            r = run_ours(sub, rank, world, local_rank)
            out[w] = {"workload": WORKLOAD_DESC[w], "value": r["value"],
                      "ms_per_step": r["ms_per_step"], "roofline_frac": r["roofline"]["frac"],
                      "steps": sub.steps, "clocks": r["clocks"],
                      "cases": [{k: c[k] for k in ("shape", "fmt", "ncols", "us_per_call",
                                                    "weight_gbps", "frac_of_measured",
                                                    "us_per_call_dependent",
                                                    "weight_gbps_dependent")}
                                for c in r["cases"]]}
        del r
        gc.collect()
        torch.cuda.empty_cache()
    out["decode_1col"] = run_decode(args, rank, world, local_rank)
    out["tensor_core"] = run_tensor_core(args, rank, world, local_rank)
    return out


def run_case_for_profile(spec: str, launches: int):
    """One case, launched `launches` times eagerly (for ncu -k/-s/-c captures).
    spec = fmt:ROWSxK:NCOLS[:tc], e.g. q6_k_planar:2560x10240:8 (":tc": with
    MMVQ_FLAG_TENSOR_CORE)."""
    import torch
    from block_quantized_matvec_gb300 import mmvq, synth
    parts = spec.split(":")
    fmt, shape, nc = parts[:3]
    flags = mmvq.FLAG_TENSOR_CORE if parts[3:] == ["tc"] else 0
    rows, K = (int(v) for v in shape.split("x"))
    nc = int(nc)
    t = {"q6_k_planar": mmvq.TYPE_Q6_K_PLANAR, "q6_k": mmvq.TYPE_Q6_K, "q4_k": mmvq.TYPE_Q4_K,
         "q4_k_planar": mmvq.TYPE_Q4_K_PLANAR, "q5_k_planar": mmvq.TYPE_Q5_K_PLANAR}[fmt]
    W = torch.from_numpy(host_weights_for(fmt, rows, K).reshape(-1)).cuda()
    if fmt.endswith("_planar"):
        W = mmvq.repack_planar(W, rows, K, type_=repack_source(fmt))
    xq = mmvq.quantize_q8_1(torch.from_numpy(synth.activations(K, nc)).cuda())
    y = torch.empty((nc, rows), device="cuda")
    for _ in range(launches):
        mmvq.gemv(t, W, rows, K, xq, nc, out=y, flags=flags)
    torch.cuda.synchronize()
    print(json.dumps({"case": spec, "launches": launches, "y0": float(y[0, 0])}))


def run_moe_case_for_profile(spec: str, launches: int):
    """The bench's MoE layer launched eagerly `launches` times (routings 100, 101,
    ...), for ncu captures.  spec = moe:T (the one-launch layer) or moe4:T (the
    same step as four launches)."""
    import torch
    from block_quantized_matvec_gb300 import mmvq, synth
    kind, T = spec.split(":")
    T = int(T)
    E, H, F, k = MOE["experts"], MOE["hidden"], MOE["ffn"], MOE["top_k"]
    dev = torch.device("cuda")
    q4 = mmvq.TYPE_Q4_K

    def planar(rows, K, salt):
        host = synth.expert_weights("q4_k", E, rows, K, salt=salt)
        per = mmvq.planar_bytes(rows, K, q4)
        out = torch.empty(E * per, dtype=torch.uint8, device=dev)
        for e in range(E):
            mmvq.repack_planar(torch.from_numpy(host[e].reshape(-1)).to(dev), rows, K,
                               out=out[e * per:(e + 1) * per], type_=q4)
        return out

    W_gu, W_dn = planar(2 * F, H, 1), planar(H, F, 2)
    x = torch.from_numpy(synth.moe_hidden(H, T)).to(dev)
    sync = mmvq.expert_ffn_workspace(dev)
    n = T * k
    for r in range(launches):
        topk = torch.from_numpy(synth.routing(T, k, E, salt=100 + r)).to(dev)
        if kind == "moe":
            mmvq.expert_ffn(mmvq.TYPE_Q4_K_PLANAR, W_gu, W_dn, E, H, F, x, topk, lists=False,
                            sync=sync)
        else:
            xq, eids, offs, act, _, st = mmvq.quantize_route_groups(x, topk, E)
            gu = mmvq.grouped(mmvq.TYPE_Q4_K_PLANAR, W_gu, E, 2 * F, H, eids, offs, act, xq, T, n,
                              status=st)
            hq = mmvq.silu_mul_quantize_q8_1(gu, F)
            mmvq.grouped(mmvq.TYPE_Q4_K_PLANAR, W_dn, E, H, F, eids, offs, None, hq, n, n,
                         status=st)
    torch.cuda.synchronize()
    print(json.dumps({"case": spec, "launches": launches}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="q6k_sweep", choices=sorted(WORKLOAD_DESC))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    help="profile mode: launch one case (fmt:ROWSxK:NCOLS, or moe:T / moe4:T for "
                         "the MoE layer in one / four launches) --launches times")
    ap.add_argument("--launches", type=int, default=8)
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload only: leave out the other workloads' summaries")
    ap.add_argument("--extra-steps", type=int, default=100,
                    help="timed steps of each extra workload of the default run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.case:
        if args.case.startswith("moe"):
            run_moe_case_for_profile(args.case, args.launches)
        else:
            run_case_for_profile(args.case, args.launches)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.workload.startswith("moe_"):
        res = run_moe(args, rank, world, local_rank)
    elif args.workload == "prologue":
        res = run_prologue(args, rank, world, local_rank)
    else:
        res = run_ours(args, rank, world, local_rank)
        if args.workload == "q6k_sweep" and not args.no_extra:
            res["workloads"] = run_extras(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
