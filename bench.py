#!/usr/bin/env python3
"""Benchmark of the CSR neighbourhood-aggregation hot path on GB300.

Default workload (one "step" = one pass of the layer set over one synthetic
input, all kernels through the C ABI):
  c2_rmat17: R-MAT scale 17 (131,072 nodes, edge factor 16, duplicates
  removed, self-loops added), X fp32 N(0,1) [N,128]; GCN SpMM (symmetric
  normalisation) + segment sum + mean + max(+argmax).
Other workloads (--workload): c3_rmat20_gatv2, c4_clustered_gt, c5_rmat22.

Prints ONE JSON line (rank 0).  Metric: aggregation Gedge*feat/s = edges x
features aggregated per second, summed over the step's layers.  Timing:
CUDA events on the launching stream around each step, L2 flushed (256 MB
write) between timed steps outside the events; max over ranks.

--impl reference times the CPU oracle (the plain single-threaded C
definition) on the host cores on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
NORTH_STAR_HBM_GBS = 8000.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the
    timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def c2_setup(torch, gnn, w):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    g = gnn.graph_prepare(dev(w["rowptr"]), dev(w["colidx"]))
    X = dev(w["X"])
    n, F = X.shape
    M = len(w["colidx"])
    outs = {k: torch.empty((n, F), dtype=torch.float32, device="cuda")
            for k in ("spmm", "sum", "mean", "max")}
    am = torch.empty((n, F), dtype=torch.int32, device="cuda")

    def step(Xin=None, events=None):
        Xs = X if Xin is None else Xin
        if events is not None:
            events["spmm"][0].record()
        gnn.gnn_spmm(g, Xs, norm=gnn.GNN_NORM_BOTH, out=outs["spmm"])
        if events is not None:
            events["spmm"][1].record()
            events["sum"][0].record()
        gnn.gnn_segment_reduce_sum(g, Xs, out=outs["sum"])
        if events is not None:
            events["sum"][1].record()
            events["mean"][0].record()
        gnn.gnn_segment_reduce_mean(g, Xs, out=outs["mean"])
        if events is not None:
            events["mean"][1].record()
            events["max"][0].record()
        gnn.gnn_segment_reduce_max(g, Xs, out=outs["max"], argmax=am)
        if events is not None:
            events["max"][1].record()

    idx = 4 * (n + 1) + 4 * M
    xb = X.numel() * X.element_size()
    yb = n * F * 4
    bcomp = {"spmm": idx + xb + yb + 8 * n, "sum": idx + xb + yb, "mean": idx + xb + yb,
             "max": idx + xb + yb + n * F * 4}
    info = {"units_per_step": 4 * M * F, "unit": "Gedge*feat/s", "dtype": "f32",
            "bcomp": bcomp, "n": n, "nnz": M, "F": F, "X": X, "outputs": list(outs.values()) + [am],
            "config": {"workload": "c2_rmat17", "graph": "R-MAT scale 17, edge factor 16, "
                       "a,b,c,d=.57,.19,.19,.05, dedup + self-loops", "nodes": n, "edges": M,
                       "features": F, "layers": ["gcn_spmm", "segment_sum", "segment_mean",
                                                 "segment_max+argmax"],
                       "mapping": "auto (degree-aware edge runs)", "l2": "flushed between steps"}}
    return step, info


def oracle_step_c2(w, rows):
    import oracle
    rp, ci, X = w["rowptr"], w["colidx"], w["X"]
    oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH, rows=rows)
    oracle.segment_reduce(oracle.OP_SUM, rp, ci, X, rows=rows)
    oracle.segment_reduce(oracle.OP_MEAN, rp, ci, X, rows=rows)
    oracle.segment_reduce(oracle.OP_MAX, rp, ci, X, rows=rows)


def sample_rows(w, frac_den=8):
    n = len(w["rowptr"]) - 1
    rows = np.arange(0, n, frac_den, dtype=np.int32)
    ne = int(np.sum(w["rowptr"][rows + 1] - w["rowptr"][rows]))
    return rows, ne


# ---------------------------------------------------------------- main

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(args):
    import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.workload(args.workload)
    rows, ne = sample_rows(w, 8)
    F = w["X"].shape[1]
    for _ in range(args.warmup):
        oracle_step_c2(w, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step_c2(w, rows)
    dt = (time.perf_counter() - t) / args.steps
    v = 4 * ne * F / dt / 1e9
    line = {"impl": "reference", "metric": "aggregation Gedge*feat/s", "value": v,
            "unit": "Gedge*feat/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "sample": f"every 8th destination row "
                       f"({len(rows)} rows, {ne} edges) per step"},
            "cpu_baseline": {"value": v, "unit": "Gedge*feat/s", "cores": 1, "kind": "oracle",
                             "sample": f"every 8th row of {args.workload}"},
            "e2e": {"value": v, "unit": "Gedge*feat/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2_rmat17")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import synth
    import sparse_neighbourhood_aggregation_gb300 as gnn

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    gnn.lib()

    w = synth.workload(args.workload)
    if args.workload != "c2_rmat17":
        raise SystemExit("only c2_rmat17 is wired into bench.py so far")
    step, info = c2_setup(torch, gnn, w)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    names = ["spmm", "sum", "mean", "max"]
    ev = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in names} for _ in range(args.steps)]
    st = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    launches0 = gnn.launch_count()
    for k in range(args.steps):
        flush.fill_(float(k))
        st[k][0].record(stream)
        step(events=ev[k])
        st[k][1].record(stream)
    torch.cuda.synchronize()
    launches = gnn.launch_count() - launches0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in st]
    total_ms = float(np.sum(step_ms))
    if world > 1:
        t = torch.tensor([total_ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms = total_ms / args.steps
    value = world * info["units_per_step"] * args.steps / (total_ms * 1e-3) / 1e9

    # per-kernel times and roofline of the dominant kernel
    hbm, _, peak_kind = measured_peaks()
    per = {k: float(np.mean([e[k][0].elapsed_time(e[k][1]) for e in ev])) for k in names}
    dom = max(per, key=per.get)
    achieved = info["bcomp"][dom] / (per[dom] * 1e-3) / 1e9
    layers = {k: {"ms": per[k], "gedge_feat_s": info["units_per_step"] / 4 / (per[k] * 1e-3) / 1e9,
                  "bcomp_bytes": info["bcomp"][k],
                  "hbm_gbs": info["bcomp"][k] / (per[k] * 1e-3) / 1e9,
                  "frac_of_measured": info["bcomp"][k] / (per[k] * 1e-3) / 1e9 / hbm,
                  "frac_of_8tbs": info["bcomp"][k] / (per[k] * 1e-3) / 1e9 / NORTH_STAR_HBM_GBS}
              for k in names}

    # end to end through the public API with host buffers
    Xh = info["X"].cpu().pin_memory()
    outs_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in info["outputs"]]
    Xdev = torch.empty_like(info["X"])
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(max(3, args.steps // 4))]
    for k, (a, b) in enumerate(e2e_ev):
        flush.fill_(float(k))
        a.record(stream)
        Xdev.copy_(Xh, non_blocking=True)
        step(Xin=Xdev)
        for oh, od in zip(outs_h, info["outputs"]):
            oh.copy_(od, non_blocking=True)
        b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in e2e_ev]))
    h2d = Xh.numel() * Xh.element_size()
    d2h = sum(o.numel() * o.element_size() for o in outs_h)

    line = {"metric": "aggregation Gedge*feat/s", "value": value, "unit": info["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": info["dtype"], "data": "synthetic", "config": info["config"],
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm,
                         "unit": "GB/s", "frac": achieved / hbm, "peak_kind": peak_kind,
                         "frac_of_8tbs": achieved / NORTH_STAR_HBM_GBS, "traffic": None,
                         "bcomp_bytes": info["bcomp"][dom]},
            "layers": layers,
            "e2e": {"value": world * info["units_per_step"] / (e2e_ms * 1e-3) / 1e9,
                    "unit": info["unit"], "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": int(launches), "clocks": clk}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle  # noqa: F401  (bench's CPU-baseline leg)
        rows, ne = sample_rows(w, 8)
        t = time.perf_counter()
        oracle_step_c2(w, rows)
        dt = time.perf_counter() - t
        line["cpu_baseline"] = {"value": 4 * ne * info["F"] / dt / 1e9, "unit": info["unit"],
                                "cores": 1, "kind": "oracle",
                                "sample": f"every 8th destination row ({len(rows)} rows, "
                                          f"{ne} edges), one step, {dt:.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
