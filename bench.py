#!/usr/bin/env python3
"""Benchmark of the fused all-gather matmul on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--sweep]

One step is one fused all-gather matmul (agmm_run) over one batch of synthetic
inputs resident in device memory; the default workload is the prefill-like
P=8, m_per_device=2048, k=8192, n=7168 problem with Y stored [n, k].

Timing: W untimed warm-up steps, then batches of exactly K steps.  Each batch
is one replay of a CUDA graph that holds exactly K steps, step i on replica
i mod R, so the inputs and outputs rotate over R replicas (footprint above
three times the L2 size: no step reads data a previous step left in L2)
whatever K is.  Each batch is bracketed by a barrier and a device synchronize
and timed with CUDA events on the stream the kernels are launched on; the
line reports the median batch (at least 7 batches, and at least a second of
timed work for the headline).  The unfused and gathered-LHS paths, and the
sub-results of the decode-like and mid-size workloads, are timed the same
way.  Rank 0 prints one JSON line.

With N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU ("replicas only": the method's exchange is between
shards that all live on one GPU here); value = all ranks' FLOPs / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused all-gather-GEMM TFLOP/s and % of roofline (tensor peak / HBM GB/s) on 1 GB300"
DEFAULT_WORKLOAD = "c4_prefill"
L2_BYTES_FALLBACK = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- distributed glue
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend: str):
    import torch.distributed as dist

    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(value: float, device=None) -> float:
    """Max of a float over ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def uniform_count(n: int, device=None) -> int:
    """The largest of the ranks' counts, on every rank: every rank must time
    the same number of barrier-bracketed batches and capture the same K."""
    return int(round(reduce_max(float(n), device)))


def batches_for(est_step_s: float, K: int, min_batches: int = 7, min_timed_s: float = 0.5,
                max_batches: int = 400) -> int:
    """Batches of K steps to time: at least min_batches and about min_timed_s
    of timed work, at most max_batches."""
    return int(min(max_batches, max(min_batches, -(-min_timed_s // max(est_step_s * K, 1e-7)))))


def steps_for(est_step_s: float, K_min: int, batch_s: float = 2e-3, K_max: int = 2000) -> int:
    """Steps per batch for a sub-result: at least K_min and about batch_s of work."""
    return int(max(K_min, min(K_max, -(-batch_s // max(est_step_s, 1e-9)))))


def aggregate_throughput(units_this_rank: float, seconds_this_rank: float, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    total = reduce_sum(units_this_rank, device)
    tmax = reduce_max(seconds_this_rank, device)
    return total / tmax, tmax


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "all_gather_gemm_agmm_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/traffic_<workload>.txt)."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha") != kernel_source_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def gpu_uuid(device) -> str:
    """nvidia-smi id of a torch device (its UUID; nvidia-smi ignores CUDA_VISIBLE_DEVICES)."""
    import torch

    u = str(getattr(torch.cuda.get_device_properties(device), "uuid", ""))
    if not u:
        return str(device.index or 0)
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- our arm
def build_replicas(w, R, device, seed=1234, dtype="bf16"):
    import torch

    tdt = torch.float16 if dtype == "f16" else torch.bfloat16

    reps = []
    g = torch.Generator(device=device)
    for r in range(R):
        g.manual_seed(seed + r)

        def draw(shape, std):
            if w.dist == "uniform":
                t = torch.rand(shape, generator=g, device=device, dtype=torch.float32) * 2 - 1
            else:
                t = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
            return t.to(tdt)

        xs = [draw((w.m_per_device, w.k), 1.0) for _ in range(w.P)]
        y = draw((w.n, w.k) if w.rhs_transpose else (w.k, w.n), 0.02)
        o = torch.empty((w.M, w.n), dtype=tdt, device=device)
        reps.append((xs, y, o))
    return reps


def capture_steps(step_fns, K, warmup, stream):
    """A CUDA graph of exactly K steps: step i runs on replica i mod R, so the
    replicas rotate inside the graph whatever K is.  W warm-up steps run
    eagerly first, then one untimed replay."""
    import torch

    R = len(step_fns)
    for i in range(max(warmup, 1)):
        step_fns[i % R](stream.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(K):
            step_fns[i % R](stream.cuda_stream)
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    return graph


def time_batches(graph, stream, batches, sampler=None):
    """Seconds of each of `batches` replays of a K-step graph, each bracketed
    by a barrier and a device synchronize, timed with events on `stream`."""
    import torch

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    times = []
    if sampler:
        sampler.start()
    for _ in range(batches):
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            graph.replay()
            end.record(stream)
        end.synchronize()
        torch.cuda.synchronize()
        barrier()
        times.append(start.elapsed_time(end) / 1000.0)
    clocks = sampler.stop() if sampler else None
    return times, clocks


def estimate_step_s(step_fns, stream, n=None):
    """Rough seconds per step from a few eager launches (sizes K and batches)."""
    import torch

    R = len(step_fns)
    n = n or max(3, min(2 * R, 50))
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(n):
            step_fns[i % R](stream.cuda_stream)
        end.record(stream)
    end.synchronize()
    return max(start.elapsed_time(end) / 1000.0 / n, 1e-7)


def measure(step_fns, K, warmup, stream, device, min_batches=7, min_timed_s=0.5, max_batches=400,
            sampler=None):
    """Median over batches of the seconds per step, K steps per batch; the
    max over ranks of each rank's median."""
    import statistics as st

    est = estimate_step_s(step_fns, stream)
    graph = capture_steps(step_fns, K, warmup, stream)
    B = uniform_count(batches_for(est, K, min_batches, min_timed_s, max_batches), device)
    times, clocks = time_batches(graph, stream, B, sampler)
    del graph
    med = st.median(times)
    med = reduce_max(med, device)
    return {"s_per_step": med / K, "K": K, "batches": B, "batch_ms_min": min(times) * 1e3,
            "batch_ms_max": max(times) * 1e3}, clocks


def cpu_oracle_sample(w, target_s=8.0, dtype="bf16"):
    """The oracle as it stands, on a bounded sample of the workload's rows."""
    import oracle
    from all_gather_gemm_agmm_gb300.inputs import make_inputs

    xs, y = make_inputs(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, w.dist, w.seed, dtype=dtype)
    rows_total = w.M
    lib = oracle.load()
    # calibrate on a block of rows, then size each call to about a second
    cal = min(rows_total, 32)
    t0 = time.perf_counter()
    oracle.agmm(xs, y, w.rhs_transpose, row_begin=0, row_end=cal, lib=lib)
    t1 = max(time.perf_counter() - t0, 1e-4) / cal
    rows = int(max(1, min(rows_total, round(1.0 / t1))))
    done_rows, spent, calls, r0 = 0, 0.0, 0, 0
    while spent < target_s and calls < 200:
        a = r0 % rows_total
        b = min(rows_total, a + rows)
        t0 = time.perf_counter()
        oracle.agmm(xs, y, w.rhs_transpose, row_begin=a, row_end=b, lib=lib)
        spent += time.perf_counter() - t0
        done_rows += b - a
        r0 = b
        calls += 1
    flops = 2.0 * done_rows * w.k * w.n
    return {"value": flops / spent / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(lib), "kind": "oracle",
            "sample": f"{done_rows} output rows of {w.name} ({rows_total} rows x {w.n} cols, k={w.k}) "
                      f"in {calls} calls, {spent:.1f} s", "seconds": spent}


def roofline_of(w, s_per_step, peaks, peak_src, sustained=False):
    """Roofline of one fused launch: algorithmic FLOPs (2*M*k*n) or unique
    bytes (2*(M*k + k*n + M*n)) over the measured seconds per launch, against
    the measured peak that bounds the shape.  A tensor-bound line takes the
    sustained bf16 peak (cuBLAS back to back for seconds, under the power cap)
    when `sustained` says its timed loop ran under the power cap too, else the
    burst peak; both fractions are reported."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = w.flops / w.unique_bytes
    if ai < ridge:
        achieved = w.unique_bytes / s_per_step / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_kind": "copy bandwidth"}
    else:
        achieved = w.flops / s_per_step / 1e12
        burst = peaks["bf16_tflops"]
        sus = peaks.get("bf16_tflops_sustained")
        use_sus = sustained and sus is not None
        peak = sus if use_sus else burst
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_kind": ("sustained: the timed loop ran under the power cap (sw_power_cap)" if use_sus
                              else "burst"),
                "frac_of_burst": achieved / burst,
                "frac_of_sustained": achieved / (sus if sus is not None else burst)}
    roof["traffic"] = recorded_traffic(w.name)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["kernel"] = "agmm_fused_sm103a"
    roof["algorithmic_bytes_per_launch"] = w.unique_bytes
    roof["flops_per_launch"] = w.flops
    roof["roofline_time_us"] = max(w.flops / (peaks["bf16_tflops"] * 1e12),
                                   w.unique_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e6
    roof["frac_of_roofline_time"] = roof["roofline_time_us"] / (s_per_step * 1e6)
    return roof


class WorkloadBench:
    """Replicas of one workload in device memory (footprint > 3x L2), a plan,
    and the step functions of the fused, unfused and gathered-LHS paths."""

    def __init__(self, w, device, dtype="bf16"):
        import torch

        import all_gather_gemm_agmm_gb300 as agmm

        self.w = w
        self.device = device
        self.l2 = torch.cuda.get_device_properties(device).L2_cache_size or L2_BYTES_FALLBACK
        self.R = max(2, -(-3 * self.l2 // w.unique_bytes))
        self.reps = build_replicas(w, self.R, device, dtype=dtype)
        self.plan = agmm.Plan(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, f16=dtype == "f16")
        self.ws = self.plan.new_workspace(False, device=device)
        self.ws_unf = self.plan.new_workspace(True, device=device)
        # inputs and zeroed workspaces come from the current stream; the
        # kernels run on another stream
        torch.cuda.synchronize()

    def fused(self):
        plan, ws, my_id = self.plan, self.ws, self.w.my_id

        def step(rep):
            xp = [x.data_ptr() for x in rep[0]]
            yp, op, wp = rep[1].data_ptr(), rep[2].data_ptr(), ws.data_ptr()
            return lambda s: plan.run_ptrs(xp, yp, op, my_id, wp, s)

        return [step(r) for r in self.reps]

    def unfused(self):
        plan, ws, my_id = self.plan, self.ws_unf, self.w.my_id
        return [(lambda rep: (lambda s: plan.run_unfused(rep[0], rep[1], rep[2], my_id, ws, s)))(r)
                for r in self.reps]

    def gathered(self):
        import torch

        plan, ws, my_id = self.plan, self.ws, self.w.my_id
        self.xcats = [torch.empty((self.w.M, self.w.k), dtype=r[2].dtype, device=self.device) for r in self.reps]
        torch.cuda.synchronize()
        return [(lambda rep, xc: (lambda s: plan.run_gather(rep[0], rep[1], rep[2], xc, my_id, ws, s)))(r, xc)
                for r, xc in zip(self.reps, self.xcats)]


def sub_result(args, name, device, stream, peaks, peak_src):
    """Fused, unfused and gathered-LHS timings of another workload, measured
    the same way as the headline (K-step graphs, median of batches); K is
    chosen so that a batch lasts at least about 2 ms."""
    import torch

    from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

    w = WORKLOADS[name]
    wb = WorkloadBench(w, device, args.dtype)
    fused = wb.fused()
    est = estimate_step_s(fused, stream)
    K = uniform_count(steps_for(est, args.steps or 20), device)
    f, _ = measure(fused, K, args.warmup, stream, device)
    wb.plan.query_status(wb.ws, stream)
    u, _ = measure(wb.unfused(), K, args.warmup, stream, device)
    wb.plan.query_status(wb.ws_unf, stream)
    g, _ = measure(wb.gathered(), K, args.warmup, stream, device)
    wb.plan.query_status(wb.ws, stream)
    roof = roofline_of(w, f["s_per_step"], peaks, peak_src)
    out = {"value": w.flops / f["s_per_step"] / 1e12 * dist_env()[0], "unit": "TFLOP/s",
           "ms_per_step": f["s_per_step"] * 1e3, "steps": K, "batches": f["batches"],
           "config": {"P": w.P, "m_per_device": w.m_per_device, "k": w.k, "n": w.n,
                      "rhs_transpose": w.rhs_transpose, "my_id": w.my_id, "replicas": wb.R,
                      "plan": wb.plan.info()},
           "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                             "roofline_time_us")},
           "unfused_ms_per_step": u["s_per_step"] * 1e3, "fused_speedup": u["s_per_step"] / f["s_per_step"],
           "with_gathered_ms_per_step": g["s_per_step"] * 1e3,
           "with_gathered_vs_unfused": u["s_per_step"] / g["s_per_step"]}
    del wb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def bench_ours(args, w):
    import torch

    import all_gather_gemm_agmm_gb300 as agmm

    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist("nccl")
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)
    wb = WorkloadBench(w, device, args.dtype)
    plan, ws = wb.plan, wb.ws
    info = plan.info()
    K = args.steps

    # the headline: the fused path, K-step graphs, median of batches, clocks
    # sampled during the timed batches
    sampler = ClockSampler(gpu_uuid(device))
    fz, clocks = measure(wb.fused(), K, args.warmup, stream, device, min_timed_s=1.0, sampler=sampler)
    plan.query_status(ws, stream)
    s_step = fz["s_per_step"]
    value = w.flops / s_step / 1e12 * ws_n  # every rank runs the same work
    ms_per_step = s_step * 1e3

    # unfused comparison and the fused path that also writes the gathered LHS
    # (what the unfused path materialises too): same replicas, same method
    uf, _ = measure(wb.unfused(), K, args.warmup, stream, device)
    plan.query_status(wb.ws_unf, stream)
    gz, _ = measure(wb.gathered(), K, args.warmup, stream, device)
    plan.query_status(ws, stream)
    unf_ms, gath_ms = uf["s_per_step"] * 1e3, gz["s_per_step"] * 1e3
    del wb.xcats

    # end to end through the C ABI from pinned host memory.  Three steps are
    # in flight: each slot has its own device buffers, plan, workspace and
    # stream, so one step's uploads overlap other steps' kernels and
    # downloads.  Every step still uploads all of its inputs and reads its O.
    # The same uploads and downloads without the kernel give the host link's
    # own time per step, the bound of this number.
    e2e = None
    if not args.no_e2e:
        reps = wb.reps
        xs_h = [x.cpu().pin_memory() for x in reps[0][0]]
        y_h = reps[0][1].cpu().pin_memory()
        n_slots = 3
        slots = []
        for si in range(n_slots):
            if si < len(reps):
                xs_d, y_d, o_d = reps[si]
            else:
                xs_d = [torch.empty_like(x) for x in reps[0][0]]
                y_d, o_d = torch.empty_like(reps[0][1]), torch.empty_like(reps[0][2])
            pl = plan if si == 0 else agmm.Plan(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose,
                                                f16=args.dtype == "f16")
            wsi = ws if si == 0 else pl.new_workspace()
            st = stream if si == 0 else torch.cuda.Stream(device=device)
            slots.append((pl, wsi, st, xs_d, y_d, o_d, torch.empty((w.M, w.n), dtype=o_d.dtype).pin_memory()))
        torch.cuda.synchronize()
        Ke = max(3, min(K, 200 if w.unique_bytes < 1e9 else 20))

        def e2e_steps(n):
            for i in range(n):
                pl, wsi, st, xs_d, y_d, o_d, o_h = slots[i % n_slots]
                pl.run_host(xs_h, y_h, o_h, xs_d, y_d, o_d, w.my_id, wsi, st)

        def link_steps(n):
            for i in range(n):
                _, _, st, xs_d, y_d, o_d, o_h = slots[i % n_slots]
                with torch.cuda.stream(st):
                    for a, b in zip(xs_d, xs_h):
                        a.copy_(b, non_blocking=True)
                    y_d.copy_(y_h, non_blocking=True)
                    o_h.copy_(o_d, non_blocking=True)

        def timed_wall(fn, n):
            fn(4)
            torch.cuda.synchronize()
            barrier()
            t0 = time.perf_counter()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(slots[0][2])
            for sl in slots[1:]:
                sl[2].wait_event(ev0)
            fn(n)
            for sl in slots[1:]:
                done = torch.cuda.Event()
                done.record(sl[2])
                slots[0][2].wait_event(done)
            ev1.record(slots[0][2])
            ev1.synchronize()
            wall = time.perf_counter() - t0
            return max(ev0.elapsed_time(ev1) / 1000.0, wall)

        e_el = timed_wall(e2e_steps, Ke)
        for pl, wsi, st, *_ in slots:
            pl.query_status(wsi, st)
        link_el = timed_wall(link_steps, Ke)
        e_val, _ = aggregate_throughput(w.flops * Ke / 1e12, e_el, device)
        e2e = {"value": e_val, "unit": "TFLOP/s", "h2d_bytes_per_step": 2 * (w.M * w.k + w.k * w.n),
               "d2h_bytes_per_step": 2 * w.M * w.n, "steps": Ke, "ms_per_step": e_el / Ke * 1e3,
               "pipelining": f"{n_slots} steps in flight ({n_slots} device buffer sets, {n_slots} streams)",
               "host_link_ms_per_step": link_el / Ke * 1e3,
               "of_host_link_bound": link_el / e_el}
        del slots, xs_h, y_h
    R, per_rep, l2 = wb.R, w.unique_bytes, wb.l2
    del wb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    subs = {}
    if not args.no_sub:
        for name in [n for n in args.sub.split(",") if n and n != w.name]:
            subs[name] = sub_result(args, name, device, stream, peaks, peak_src)
    sweep_smp = None if args.no_sub else sweep_sample(args, device, stream, peaks, peak_src)

    roof = roofline_of(w, s_step, peaks, peak_src,
                       sustained="sw_power_cap" in (clocks or {}).get("reasons", []))
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws_n, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.dtype, "data": "synthetic (seeded torch.Generator on device; shapes of the workload)",
        "config": {"workload": w.name, "P": w.P, "m_per_device": w.m_per_device, "k": w.k, "n": w.n,
                   "rhs_transpose": w.rhs_transpose, "my_id": w.my_id, "dist": w.dist,
                   "l2": f"inputs larger than L2: {R} rotating input/output replicas, "
                         f"{R * per_rep / 2**20:.0f} MiB > 3x L2 ({l2 / 2**20:.0f} MiB)",
                   "timing": f"median of {fz['batches']} batches, each one replay of a CUDA graph of exactly "
                             f"{K} steps (step i on replica i mod {R}), events on the launch stream, "
                             "barrier and synchronize around each batch; max over ranks",
                   "batch_ms_range": [fz["batch_ms_min"], fz["batch_ms_max"]],
                   "parallelism": f"replicas x{ws_n}", "plan": info},
        "roofline": roof,
        "unfused": {"ms_per_step": unf_ms, "value": w.flops / (unf_ms / 1e3) / 1e12 * ws_n, "steps": K,
                    "batches": uf["batches"], "fused_speedup": unf_ms / ms_per_step},
        "with_gathered": {"ms_per_step": gath_ms, "steps": K, "batches": gz["batches"],
                          "vs_unfused": unf_ms / gath_ms, "cost_over_fused": gath_ms / ms_per_step},
        "sub_results": subs,
        "sweep_sample": sweep_smp,
        "e2e": e2e,
        "gpu_launches": K,
        "gpu_launches_note": "fused kernel launches per timed batch (one per step)",
        "clocks": clocks,
    }
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_oracle_sample(w, target_s=args.cpu_seconds, dtype=args.dtype)
    if rank == 0:
        print(json.dumps(result), flush=True)


SWEEP_SAMPLE = ("sweep_P2_m8_rt", "sweep_P8_m8_nt", "sweep_P4_m32_rt", "sweep_P2_m128_nt", "sweep_P8_m128_rt",
                "sweep_P2_m1000_rt", "sweep_P4_m1000_nt", "sweep_P8_m4096_nt")


def sweep_sample(args, device, stream, peaks, peak_src):
    """Fused against gather-then-GEMM on a sample of the sweep spanning its P,
    m and layouts, timed like the headline (K-step graphs over replicas larger
    than L2, median of at least 7 batches) with shorter timed regions."""
    import torch

    from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

    points = []
    for name in [n for n in args.sweep_sample.split(",") if n]:
        w = WORKLOADS[name]
        wb = WorkloadBench(w, device, args.dtype)
        fused = wb.fused()
        K = uniform_count(steps_for(estimate_step_s(fused, stream), args.steps or 20), device)
        f, _ = measure(fused, K, args.warmup, stream, device, min_timed_s=0.15)
        wb.plan.query_status(wb.ws, stream)
        u, _ = measure(wb.unfused(), K, args.warmup, stream, device, min_timed_s=0.15)
        wb.plan.query_status(wb.ws_unf, stream)
        roof = roofline_of(w, f["s_per_step"], peaks, peak_src)
        points.append({"point": name.replace("sweep_", ""), "fused_us": f["s_per_step"] * 1e6,
                       "unfused_us": u["s_per_step"] * 1e6, "fused_speedup": u["s_per_step"] / f["s_per_step"],
                       "bound": roof["bound"], "frac": roof["frac"], "steps": K, "batches": f["batches"]})
        del wb, fused
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return {"points": points, "fused_faster_everywhere": all(q["fused_speedup"] > 1.0 for q in points),
            "timing": "per point: K-step CUDA graphs over replicas > 3x L2, median of >= 7 batches, "
                      "fused and unfused on the same replicas; max over ranks"}


def bench_sweep(args):
    """Fused vs unfused device time at every point of the k=5120, n=2560
    sweep, each timed like the headline (K-step graphs, median of batches)."""
    import torch

    from all_gather_gemm_agmm_gb300.inputs import SWEEP

    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=device)
    names = set(args.sweep_points.split(",")) if args.sweep_points else None
    for w in SWEEP:
        if names and w.name not in names:
            continue
        wb = WorkloadBench(w, device, args.dtype)
        fused = wb.fused()
        est = estimate_step_s(fused, stream)
        K = steps_for(est, args.steps or 20)
        f, _ = measure(fused, K, args.warmup, stream, device)
        wb.plan.query_status(wb.ws, stream)
        u, _ = measure(wb.unfused(), K, args.warmup, stream, device)
        wb.plan.query_status(wb.ws_unf, stream)
        f_us, u_us = f["s_per_step"] * 1e6, u["s_per_step"] * 1e6
        roof = roofline_of(w, f["s_per_step"], peaks, peak_src)
        print(json.dumps({"sweep_point": w.name, "P": w.P, "m_per_device": w.m_per_device,
                          "rhs_transpose": w.rhs_transpose, "fused_us": f_us, "unfused_us": u_us,
                          "fused_tflops": w.flops / (f_us * 1e-6) / 1e12, "roofline_us": roof["roofline_time_us"],
                          "bound": roof["bound"], "frac": roof["frac"],
                          "frac_of_roofline": roof["frac_of_roofline_time"], "fused_faster": f_us < u_us,
                          "steps": K, "batches": f["batches"], "plan": wb.plan.info()}), flush=True)
        del wb, fused
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def bench_profile_target(args, w):
    """A plain run for profilers: W warm-up launches, then K launches of one
    path (--path fused | unfused | gather) over the workload's replicas, eager
    (no CUDA graph), then a status check.  Prints nothing timed: a number
    taken under a profiler is not a benchmark value."""
    import torch

    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=device)
    wb = WorkloadBench(w, device, args.dtype)
    fns = {"fused": wb.fused, "unfused": wb.unfused, "gather": wb.gathered}[args.path]()
    for i in range(args.warmup + args.steps):
        fns[i % len(fns)](stream.cuda_stream)
    wb.plan.query_status(wb.ws_unf if args.path == "unfused" else wb.ws, stream)
    torch.cuda.synchronize()
    print(json.dumps({"profile_target": w.name, "path": args.path, "launches": args.warmup + args.steps,
                      "replicas": wb.R, "plan": wb.plan.info()}), flush=True)


# ----------------------------------------------------------------------------- reference arm
def bench_reference(args, w):
    """The oracle as it stands, on the host cores, on bounded samples of the
    same workload: each step computes a block of output rows."""
    ws_n, rank, _ = dist_env()
    if ws_n > 1 and rank != 0:
        return
    import oracle
    from all_gather_gemm_agmm_gb300.inputs import make_inputs

    xs, y = make_inputs(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, w.dist, w.seed, dtype=args.dtype)
    lib = oracle.load()
    cal = min(w.M, 32)
    t0 = time.perf_counter()
    oracle.agmm(xs, y, w.rhs_transpose, row_begin=0, row_end=cal, lib=lib)
    t_row = max(time.perf_counter() - t0, 1e-4) / cal
    rows = int(max(1, min(w.M, round(args.ref_step_seconds / t_row))))
    for i in range(args.warmup):
        oracle.agmm(xs, y, w.rhs_transpose, row_begin=0, row_end=rows, lib=lib)
    K = args.steps or 5
    t0 = time.perf_counter()
    for i in range(K):
        a = (i * rows) % max(1, w.M - rows + 1)
        oracle.agmm(xs, y, w.rhs_transpose, row_begin=a, row_end=a + rows, lib=lib)
    el = time.perf_counter() - t0
    flops = 2.0 * rows * w.k * w.n * K
    val = flops / el / 1e12
    sample = f"{rows} of {w.M} output rows of {w.name} per step"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": ws_n, "steps": K,
        "warmup": args.warmup, "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded torch.Generator on the CPU)",
        "config": {"workload": w.name, "P": w.P, "m_per_device": w.m_per_device, "k": w.k, "n": w.n,
                   "rhs_transpose": w.rhs_transpose, "my_id": w.my_id},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.max_threads(lib), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="steps per timed batch (one K-step CUDA graph)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true", help="fused vs unfused at every sweep point")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sub", action="store_true", help="skip the other workloads' sub-results")
    ap.add_argument("--sub", default="c2_decode,c3_mid",
                    help="comma-separated workloads measured as sub-results of the same line")
    ap.add_argument("--sweep-points", default="", help="with --sweep: comma-separated sweep point names")
    ap.add_argument("--sweep-sample", default=",".join(SWEEP_SAMPLE),
                    help="sweep points timed fused against unfused in the default run ('' for none)")
    ap.add_argument("--profile-target", action="store_true",
                    help="only launch W + K steps of --path, eagerly, for a profiler (no timing)")
    ap.add_argument("--path", choices=["fused", "unfused", "gather"], default="fused")
    ap.add_argument("--dtype", choices=["bf16", "f16"], default="bf16",
                    help="element type of X, Y and O (fp16: the tutorial's float16 variant)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--ref-step-seconds", type=float, default=1.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        bench_reference(args, w)
    elif args.profile_target:
        bench_profile_target(args, w)
    elif args.sweep:
        bench_sweep(args)
    else:
        bench_ours(args, w)


if __name__ == "__main__":
    main()
