"""Autotuner of the tile configuration, and the writer of the tuned table.

all_gather_matmul (tpu_inference "all_gather_matmul.py") looks its block
sizes up in a table of tuned sizes keyed by shape, dtype and mesh size
(get_tuned_block_sizes) and falls back to defaults for shapes it lacks.  The
planner of libagmm.so does the same with ``csrc/tuned_sm103.inc``: an
``agmm_tile_config_t`` per exact (P, m_per_device, k, n, rhs_transpose,
input type), else its own rules.  This module measures candidate
configurations on the GPU and writes that table:

    python -m all_gather_gemm_agmm_gb300.tune --out results.json [--workloads c2_decode,...]
    python -m all_gather_gemm_agmm_gb300.tune --emit results.json   # rewrites csrc/tuned_sm103.inc

Each shape's candidates are distinct plans (configurations that yield the
same plan are timed once).  Every candidate's output is checked against the
planner's own choice before it is timed.  Timing follows the benchmark's
rules: a CUDA graph of launches over input replicas whose footprint exceeds
three times L2, timed with CUDA events on the launch stream.  A screening
pass times every candidate briefly; the fastest few and the planner's choice
are then timed again, interleaved, and a configuration enters the table only
when it beats the planner's choice by at least ``MARGIN``.
"""
from __future__ import annotations

import argparse
import datetime
import itertools
import json
import math
import os
import sys
from typing import Dict, List, Optional, Sequence, Tuple

from . import AgmmError, CONFIG_FIELDS, PKG_DIR, Plan, plan_preview, tile_config
from .inputs import SWEEP, WORKLOADS, Workload

TABLE_PATH = os.path.join(PKG_DIR, "csrc", "tuned_sm103.inc")
MARGIN = 0.02  # a tuned entry must be at least 2 % faster than the planner's rules
_NO_TABLE = {"tuned_table": False}

_INC_HEADER = """\
// Tuned tile configurations for GB300 (sm_103a), one per exact shape:
// {P, m_per_device, k, n, rhs_transpose, fp16, {path, chunks, box_rows,
// tile_n, cluster_m, cta_pair, stages, group_m, stream_k, row_groups, splits,
// dsmem_reduce, tuned_table}}.  Written by tune.py; do not edit by hand.
"""


def _plan_key(info: Dict[str, int]) -> Tuple:
    """What makes two plans the same kernel launch."""
    return tuple(info[f] for f in ("path", "box_rows", "whole_shards", "tile_n", "stages", "splits", "num_ctas",
                                   "group_m", "row_groups", "cluster_m", "cta_pair", "stream_k_tiles",
                                   "dsmem_reduce", "k_blocks_per_stage"))


def candidates(P: int, m: int, k: int, n: int, rt: bool, f16: bool = False, num_sms: int = 152) -> List[Dict]:
    """Candidate configurations for one shape, checked on the host
    (agmm_plan_preview): those the planner accepts, each a distinct preview."""
    base = plan_preview(P, m, k, n, rt, num_sms=num_sms, f16=f16, config=_NO_TABLE)
    raw: List[Dict] = [dict(_NO_TABLE)]
    swap_ok = True
    try:
        plan_preview(P, m, k, n, rt, num_sms=num_sms, f16=f16, config={"path": "swap", "tuned_table": False})
    except AgmmError:
        swap_ok = False
    if swap_ok:
        n_tiles = n // 128
        for chunks in ("half", "whole"):
            for G in (1, 2, 4, 8):
                s_auto = max(1, min(16, num_sms // (n_tiles * G), k // 64))
                for S in sorted({s_auto, max(1, (3 * s_auto) // 4), max(1, s_auto // 2)}):
                    raw.append({"path": "swap", "chunks": chunks, "row_groups": G, "splits": S, "tuned_table": False})
        raw.append({"path": "swap", "dsmem_reduce": True, "tuned_table": False})
    # row tiles (for shapes that fit swapped tiles, only their main variants)
    tile_ns = [256, 128] if n % 256 == 0 else [128]
    # (a two-CTA cluster always multiplies as a CTA pair)
    variants = itertools.product(tile_ns, (2, 1), (True, False), (4, 8, 16))
    if swap_ok:
        variants = itertools.product(tile_ns, (2, 1), (True,), (8,))
    for bn, cm, sk, gm in variants:
        raw.append({"path": "rows", "tile_n": bn, "cluster_m": cm, "cta_pair": cm == 2, "stream_k": sk,
                    "group_m": gm, "tuned_table": False})
    out, seen = [], set()
    for cfg in raw:
        try:
            info = plan_preview(P, m, k, n, rt, num_sms=num_sms, f16=f16, config=cfg)
        except AgmmError:
            continue
        key = _plan_key(info)
        if key in seen:
            continue
        seen.add(key)
        out.append(cfg)
    assert out and out[0] == _NO_TABLE, base
    return out


class _Bench:
    """Input replicas of one shape on the GPU, and a timer for plans over them."""

    def __init__(self, w: Workload, f16: bool = False, seed: int = 4321):
        import torch

        self.torch = torch
        self.w, self.f16 = w, f16
        dev = torch.device("cuda", torch.cuda.current_device())
        self.dt = torch.float16 if f16 else torch.bfloat16
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.R = max(2, math.ceil(3 * l2 / w.unique_bytes))
        g = torch.Generator(device=dev)
        self.reps = []
        for r in range(self.R):
            g.manual_seed(seed + r)

            def draw(shape, std):
                if w.dist == "uniform":
                    t = torch.rand(shape, generator=g, device=dev, dtype=torch.float32) * 2 - 1
                else:
                    t = torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std
                return t.to(self.dt)

            xs = [draw((w.m_per_device, w.k), 1.0) for _ in range(w.P)]
            y = draw((w.n, w.k) if w.rhs_transpose else (w.k, w.n), 0.02)
            o = torch.empty((w.M, w.n), dtype=self.dt, device=dev)
            self.reps.append((xs, y, o))
        self.stream = torch.cuda.Stream()
        self.reference: Optional["torch.Tensor"] = None

    def plan(self, cfg: Dict) -> Plan:
        w = self.w
        return Plan(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, f16=self.f16, config=cfg)

    def check(self, plan: Plan, ws) -> bool:
        """Run replica 0 once; compare with the first checked plan's output."""
        torch = self.torch
        xs, y, o = self.reps[0]
        with torch.cuda.stream(self.stream):  # poison on the launch stream: a skipped store stays NaN
            o.fill_(float("nan"))
        plan.run(xs, y, o, self.w.my_id, ws, self.stream.cuda_stream)
        plan.query_status(ws, self.stream.cuda_stream)
        self.stream.synchronize()
        got = o.float()
        if self.reference is None:
            self.reference = got.clone()
            return bool(torch.isfinite(got).all())
        err = (got - self.reference).norm() / self.reference.norm().clamp_min(1e-30)
        return bool(torch.isfinite(got).all()) and float(err) <= 5e-3

    def capture(self, plan: Plan, ws):
        torch = self.torch
        fns = [(lambda r: (lambda s: plan.run(r[0], r[1], r[2], self.w.my_id, ws, s)))(r) for r in self.reps]
        for i in range(3):
            fns[i % self.R](self.stream.cuda_stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            for fn in fns:
                fn(self.stream.cuda_stream)
        with torch.cuda.stream(self.stream):
            graph.replay()
        torch.cuda.synchronize()
        return graph

    def time(self, graph, seconds: float) -> float:
        """Microseconds per launch over about `seconds` of whole graph replays."""
        torch = self.torch
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            start.record(self.stream)
            graph.replay()
            end.record(self.stream)
        end.synchronize()
        one = max(start.elapsed_time(end) / 1e3, 1e-6)
        reps = max(1, int(round(seconds / one)))
        with torch.cuda.stream(self.stream):
            start.record(self.stream)
            for _ in range(reps):
                graph.replay()
            end.record(self.stream)
        end.synchronize()
        return start.elapsed_time(end) * 1e3 / (reps * self.R)


def tune_shape(w: Workload, f16: bool = False, screen_s: float = 0.04, final_s: float = 0.15, finalists: int = 3,
               rounds: int = 3, log=None) -> Dict:
    """Time every candidate of one shape; return the record the table is
    written from (the planner's choice, the fastest candidate, all trials)."""
    torch_bench = _Bench(w, f16)
    torch = torch_bench.torch
    cands = candidates(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, f16=f16,
                       num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
    trials, live, seen = [], [], set()
    for cfg in cands:
        rec = {"config": {k: v for k, v in cfg.items() if k != "tuned_table"}}
        try:
            plan = torch_bench.plan(cfg)
        except AgmmError as e:
            rec["error"] = str(e)
            trials.append(rec)
            continue
        info = plan.info()
        key = _plan_key(info)
        if key in seen:  # the device lowered it onto a plan already timed
            plan.close()
            continue
        seen.add(key)
        ws = plan.new_workspace()
        torch.cuda.synchronize()
        try:
            ok = torch_bench.check(plan, ws)
        except AgmmError as e:
            ok, rec["error"] = False, str(e)
        rec["plan"] = {f: info[f] for f in ("path", "box_rows", "whole_shards", "tile_n", "stages", "splits",
                                            "num_ctas", "group_m", "row_groups", "cluster_m", "cta_pair",
                                            "stream_k_tiles", "dsmem_reduce")}
        if not ok:
            rec.setdefault("error", "output differs from the planner's choice")
            trials.append(rec)
            plan.close()
            continue
        graph = torch_bench.capture(plan, ws)
        rec["screen_us"] = round(torch_bench.time(graph, screen_s), 3)
        plan.query_status(ws, torch_bench.stream)
        trials.append(rec)
        live.append((rec, plan, ws, graph))
        if log:
            log(f"  {w.name}: {rec['screen_us']:9.2f} us  {rec['config']}")
    # final round: the planner's choice and the fastest few, interleaved
    heuristic = live[0]
    order = sorted(live[1:], key=lambda t: t[0]["screen_us"])[:finalists]
    final = [heuristic] + order
    times = {id(t[0]): [] for t in final}
    for _ in range(rounds):
        for t in final:
            times[id(t[0])].append(torch_bench.time(t[3], final_s))
    for t in final:
        ts = sorted(times[id(t[0])])
        t[0]["final_us"] = round(ts[len(ts) // 2], 3)
    for rec, plan, ws, graph in live:
        plan.query_status(ws, torch_bench.stream)
    best = min(final, key=lambda t: t[0]["final_us"])[0]
    h = heuristic[0]
    chosen = best is not h and best["final_us"] <= h["final_us"] * (1.0 - MARGIN)
    out = {
        "name": w.name, "P": w.P, "m_per_device": w.m_per_device, "k": w.k, "n": w.n,
        "rhs_transpose": bool(w.rhs_transpose), "f16": bool(f16),
        "rules": {"plan": h["plan"], "us": h["final_us"]},
        "best": {"config": best["config"], "plan": best["plan"], "us": best["final_us"]},
        "tuned": bool(chosen),
        "trials": [{k: v for k, v in t.items() if k != "plan"} for t in trials],
    }
    del live, final, heuristic, order
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def _inc_value(field: str, v) -> int:
    return int(tile_config({field: v}).__getattribute__(field))


def emit(results: Sequence[Dict], path: str = TABLE_PATH) -> str:
    """Write the table of the records whose tuned configuration won; returns
    the text written."""
    lines = [_INC_HEADER]
    for r in sorted(results, key=lambda r: (r["P"], r["m_per_device"], r["k"], r["n"], r["rhs_transpose"],
                                          r["f16"])):
        if not r.get("tuned"):
            continue
        cfg = dict(r["best"]["config"])
        tc = tile_config(cfg)
        vals = ", ".join(str(getattr(tc, f)) for f in CONFIG_FIELDS)
        lines.append("{%d, %d, %d, %d, %d, %d, {%s}},  // %s: %.2f -> %.2f us\n" % (
            r["P"], r["m_per_device"], r["k"], r["n"], int(r["rhs_transpose"]), int(r["f16"]), vals, r["name"],
            r["rules"]["us"], r["best"]["us"]))
    text = "".join(lines)
    with open(path, "w") as f:
        f.write(text)
    return text


def write_records(doc: Dict, path: str) -> None:
    """The records file: its header fields, then one record per line."""
    head = {k: v for k, v in doc.items() if k != "records"}
    body = ",\n".join(json.dumps(r, separators=(",", ":")) for r in doc["records"])
    with open(path, "w") as f:
        f.write(json.dumps(head)[:-1] + ', "records": [\n' + body + "\n]}\n")


def _workloads(spec: str) -> List[Workload]:
    if spec == "all":
        return [WORKLOADS[n] for n in ("c1_tiny", "c2_decode", "c3_mid", "c4_prefill")] + list(SWEEP)
    return [WORKLOADS[n] for n in spec.split(",") if n]


def main(argv: Optional[Sequence[str]] = None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workloads", default="all", help="comma-separated workload names, or 'all'")
    ap.add_argument("--f16", action="store_true", help="tune the fp16 variant of each shape")
    ap.add_argument("--out", help="write the tuning records (JSON) here")
    ap.add_argument("--emit", metavar="JSON", help="rewrite the tuned table from a records file and exit")
    ap.add_argument("--table", default=TABLE_PATH, help="table path for --emit")
    args = ap.parse_args(argv)
    if args.emit:
        with open(args.emit) as f:
            emit(json.load(f)["records"], args.table)
        return 0
    import torch

    if not torch.cuda.is_available():
        print("tune: no CUDA device", file=sys.stderr)
        return 2
    records = []
    for w in _workloads(args.workloads):
        rec = tune_shape(w, f16=args.f16, log=lambda s: print(s, file=sys.stderr, flush=True))
        records.append(rec)
        print(json.dumps({k: rec[k] for k in ("name", "rules", "best", "tuned")}), flush=True)
        if args.out:  # rewritten after every shape, so a cut-off run keeps what it measured
            props = torch.cuda.get_device_properties(0)
            doc = {"device": props.name, "sms": props.multi_processor_count,
                   "date": datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%d"),
                   "command": "python -m all_gather_gemm_agmm_gb300.tune " + " ".join(argv or sys.argv[1:]),
                   "margin": MARGIN, "records": records}
            write_records(doc, args.out)
    return 0


if __name__ == "__main__":
    sys.exit(main())
