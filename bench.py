#!/usr/bin/env python3
"""Benchmark of the CSR neighbourhood-aggregation hot path on GB300.

Every kernel is launched through the C ABI (include/gnn.h) by the Python
binding.  With no --workload the run measures, in one process and one JSON
line:

  headline step, c5_rmat22: GCN SpMM (symmetric normalisation) on R-MAT
      scale 22 (4,194,304 nodes, edge factor 16, a,b,c,d = .57,.19,.19,.05,
      duplicates removed, self-loops added), X bf16 N(0,1) [N,256], fp32
      accumulation and output, original vertex ids, AUTO (edge-span)
      mapping -- the largest power-law graph of the workloads;
  families, each on its own graph and timed the same way:
    c2_rmat17: R-MAT scale 17, X fp32 N(0,1) [N,128]: SpMM, segment sum,
        mean and max (+argmax);
    c3_rmat20_gatv2: R-MAT scale 20, H bf16 [N,256], W bf16 [256,256],
        4 heads x 64: the fused GATv2 layer (tcgen05 projection + fused
        score / online softmax / aggregate), the projection alone, and the
        attention by difference;
    c4_clustered_gt: clustered graph 1024 x 256 nodes (p = 0.3, 1% rewired),
        Q, K, V bf16 [N, 8x32]: Graph Transformer attention on the backend
        the adaptive selector picks (and the CSR path beside it).

--workload NAME runs one workload alone (c2_rmat17, c3_rmat20_gatv2,
c4_clustered_gt, c4_clustered_spmm, c5_rmat22; --mapping / --ordering for
the c5 study, --tiles for the c4 tile paths, --features for c2).

Metric: aggregation Gedge*feat/s = edges x features aggregated per second
(attention: edges x heads x head_dim).  Timing: CUDA events on the
launching stream around every layer, an L2 flush (a 512 MB write, outside
the events) before EVERY timed layer ("cold"); median, min and mean over the
K steps; "warm" = the same layer K times back to back with no flush (the
second-pass cache mode); for the scale-17 layers also "warm_graph", 20
back-to-back calls captured in one CUDA graph and replayed, per call.  Max
over ranks.  e2e: the headline step through the same API starting from
pinned host buffers, every step copying its inputs in and reading its
results back inside the timed region, steps pipelined over three streams
(copy in, compute, read back; the sequential per-step figure beside it).
The roofline object describes
the headline step's dominant kernel: achieved = its compulsory bytes
(indices read once, every feature row read once, every output written
once) / its mean event-timed duration; traffic = the DRAM bytes of an ncu
capture recorded for the same kernel sources, else null.

--impl reference times the CPU oracle (plain single-threaded C, fp64) on a
bounded sample of destination rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
METRIC = "aggregation Gedge*feat/s"
UNIT = "Gedge*feat/s"
HEADLINE = "c5_rmat22"
FAMILIES = ("c2_rmat17", "c3_rmat20_gatv2", "c4_clustered_gt")
CSRC = os.path.join(ROOT, "sparse_neighbourhood_aggregation_gb300", "csrc")
# kernel sources whose ncu DRAM counters a recorded traffic figure covers
TRAFFIC_SOURCES = {"spmm": ("aggregate.cu", "common.cuh", "runtime.cu"),
                   "sum": ("aggregate.cu", "common.cuh", "runtime.cu"),
                   "mean": ("aggregate.cu", "common.cuh", "runtime.cu"),
                   "max": ("aggregate.cu", "common.cuh", "runtime.cu")}
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.md")


def sources_sha16(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, layer: str):
    """DRAM bytes (read + write) per launch of `layer` on `workload` from the
    recorded ncu table, or None when no capture exists or the kernel sources
    changed since it was taken (their hash differs)."""
    files = TRAFFIC_SOURCES.get(layer)
    if not files or not os.path.exists(TRAFFIC_TABLE):
        return None, None
    sha = sources_sha16(files)
    with open(TRAFFIC_TABLE) as f:
        for ln in f:
            cells = [c.strip() for c in ln.strip().strip("|").split("|")]
            if len(cells) >= 4 and cells[0] == workload and cells[1] == layer:
                try:
                    val = float(cells[2])
                except ValueError:
                    continue
                if cells[3] == sha:
                    return val, sha
                return None, sha
    return None, sha


def host_cpu():
    """CPU model and logical core count of this host (for the CPU baseline)."""
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return model, os.cpu_count()


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

class Layer:
    """One API call of the step: fn(inputs) launches it; units = edge x
    feature products it aggregates; bcomp = its compulsory bytes."""

    def __init__(self, name, fn, units, bcomp, bound="hbm"):
        self.name, self.fn, self.units, self.bcomp, self.bound = name, fn, units, bcomp, bound


class Workload:
    def __init__(self, name, layers, inputs, outputs, config, dtype, oracle_step, sample_rows,
                 extra=None):
        self.name = name
        self.layers = layers
        self.inputs = inputs        # device tensors a step reads (copied from host in e2e)
        self.outputs = outputs      # device tensors a step writes (read back in e2e)
        self.config = config
        self.dtype = dtype
        self.oracle_step = oracle_step
        self.sample_rows = sample_rows
        self.extra = extra or {}

    def step(self, ins=None):
        ins = self.inputs if ins is None else ins
        for L in self.layers:
            L.fn(ins)


def _dev(torch, a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _sample_by_edges(rp, target_edges, seed=0):
    """Destination rows in a fixed random order until ~target_edges edges."""
    n = len(rp) - 1
    order = np.random.default_rng(seed).permutation(n)
    cum = np.cumsum(np.diff(rp)[order])
    k = int(np.searchsorted(cum, target_edges)) + 1
    rows = np.sort(order[:k]).astype(np.int32)
    return rows, int(np.sum(rp[rows + 1] - rp[rows]))


def selector_report(torch, gnn, g, op, dtype, F=0, heads=0, head_dim=0):
    """Graph statistics measured on the GPU (degree moments, local density)
    and the backend the rule picks for op; the statistics pass is timed on
    the host clock around the synchronous call (prep, not in a step)."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = gnn.gnn_graph_stats_compute(g)
    ms = (time.perf_counter() - t0) * 1e3
    backend, thr = gnn.gnn_select_backend(st, op, dtype, F, heads, head_dim)
    return {"stats_ms": ms, "max_degree": st.max_degree, "mean_degree": st.mean_degree,
            "degree_std": st.degree_std, "degree_skewness": st.degree_skewness,
            "listed_blocks": st.n_blocks, "edges_per_block": st.edges_per_block,
            "backend": "tiles" if backend == gnn.GNN_BACKEND_TILES else "csr",
            "fill_threshold": thr if backend == gnn.GNN_BACKEND_TILES else None}


def setup_c2(torch, gnn, w):
    g = gnn.graph_prepare(_dev(torch, w["rowptr"]), _dev(torch, w["colidx"]))
    X = _dev(torch, w["X"])
    n, F = X.shape
    M = len(w["colidx"])
    outs = {k: torch.empty((n, F), dtype=torch.float32, device="cuda")
            for k in ("spmm", "sum", "mean", "max")}
    am = torch.empty((n, F), dtype=torch.int32, device="cuda")
    idx = 4 * (n + 1) + 4 * M
    xb, yb = X.numel() * X.element_size(), n * F * 4
    layers = [
        Layer("spmm", lambda ins: gnn.gnn_spmm(g, ins[0], norm=gnn.GNN_NORM_BOTH,
                                               out=outs["spmm"]), M * F, idx + xb + yb + 8 * n),
        Layer("sum", lambda ins: gnn.gnn_segment_reduce_sum(g, ins[0], out=outs["sum"]), M * F,
              idx + xb + yb),
        Layer("mean", lambda ins: gnn.gnn_segment_reduce_mean(g, ins[0], out=outs["mean"]), M * F,
              idx + xb + yb),
        Layer("max", lambda ins: gnn.gnn_segment_reduce_max(g, ins[0], out=outs["max"],
                                                            argmax=am), M * F,
              idx + xb + yb + n * F * 4),
    ]

    def oracle_step(rows):
        import oracle
        rp, ci, Xh = w["rowptr"], w["colidx"], w["X"]
        oracle.spmm(rp, ci, Xh, norm=oracle.NORM_BOTH, rows=rows)
        oracle.segment_reduce(oracle.OP_SUM, rp, ci, Xh, rows=rows)
        oracle.segment_reduce(oracle.OP_MEAN, rp, ci, Xh, rows=rows)
        oracle.segment_reduce(oracle.OP_MAX, rp, ci, Xh, rows=rows)

    # rows narrower than 32 16-byte chunks (e.g. F = 32 fp32) run on the
    # sub-warp workers of the generic kernel: its own workload name
    name = "c2_rmat17" if F == 128 else f"c2_rmat17_f{F}"
    cfg = {"workload": name, "graph": "R-MAT scale 17, edge factor 16, "
           "a,b,c,d=.57,.19,.19,.05, dedup + self-loops", "nodes": n, "edges": M, "features": F,
           "x_dtype": "fp32", "layers": ["gcn_spmm", "segment_sum", "segment_mean",
                                         "segment_max+argmax"],
           "mapping": "auto (degree-aware edge runs)"}
    # ~4 x 8.3M edge-rows of oracle work (all rows): ~10 s on one core
    rows = np.arange(n, dtype=np.int32)
    # segment min + argmin, the pages' own degree-aware reduction (timed
    # apart: the configured step is SpMM, sum, mean, max)
    ymin = torch.empty((n, F), dtype=torch.float32, device="cuda")
    amin = torch.empty((n, F), dtype=torch.int32, device="cuda")
    # backward of max through its argmax (grad_out, argmax read; grad_X written)
    gout = torch.randn((n, F), dtype=torch.float32, device="cuda")
    gx = torch.empty((n, F), dtype=torch.float32, device="cuda")
    timed = {
        "segment_min_argmin": (lambda: gnn.gnn_segment_reduce_min(g, X, out=ymin, argmin=amin),
                               idx + xb + yb + n * F * 4, "timed apart, cold", M * F),
        "max_backward": (lambda: gnn.gnn_segment_reduce_ext_backward(am, gout, n, out=gx),
                         3 * n * F * 4, "argmax scatter of grad_out into grad_X (zero-fill "
                                        "included), timed apart, cold"),
        "csr_transpose": (lambda: gnn.gnn_csr_transpose(g), 0,
                          "CSR^T build (count, stable radix sort, scan), timed apart, cold; the "
                          "SpMM backward is a SpMM on it"),
    }
    return Workload(name, layers, [X], list(outs.values()) + [am], cfg, "f32",
                    oracle_step, (rows, M), extra={"timed": timed,
                                                  "selector": selector_report(
                                                      torch, gnn, g, gnn.GNN_OP_SPMM, gnn.GNN_F32, F)})


def setup_c3(torch, gnn, w):
    g = gnn.graph_prepare(_dev(torch, w["rowptr"]), _dev(torch, w["colidx"]))
    H = _dev(torch, w["H"])
    W = _dev(torch, w["W"])
    a = _dev(torch, w["a"])
    n = H.shape[0]
    M = len(w["colidx"])
    heads, D = w["heads"], w["head_dim"]
    HD = heads * D
    out = torch.empty((n, HD), dtype=torch.float32, device="cuda")
    lse = torch.empty((n, heads), dtype=torch.float32, device="cuda")
    C = torch.empty((n, HD), dtype=torch.bfloat16, device="cuda")
    idx = 4 * (n + 1) + 4 * M
    # fused layer: H read, C written then read once, out + lse written, indices read
    b_proj = n * 256 * 2 + n * HD * 2 + 256 * HD * 2 + n * heads * 4
    b_attn = idx + n * HD * 2 + n * HD * 4 + n * heads * 4 + 2 * n * heads * 4
    layers = [Layer("gatv2_fwd", lambda ins: gnn.gnn_gatv2_fwd(g, ins[0], W, a, heads, D,
                                                               w["slope"], out=out, lse=lse),
                    M * HD, b_proj + b_attn, "alu")]

    def proj_only():
        gnn.gnn_projection(H, W, out=C)

    def oracle_step(rows):
        import oracle
        oracle.gatv2(w["rowptr"], w["colidx"], w["H"], w["W"], w["a"], heads, D, w["slope"],
                     rows=rows)

    # backward of the attention (AL over CSR, R over CSR^T, attention-vector
    # reduction) from the timed forward's out and lse; C = H W as the forward
    # scored it; compulsory bytes: C read by each kernel, dO by each, O once,
    # dl and dr written, lse and G read twice / written once, both index sets
    rpt, cit, _ = gnn.gnn_csr_transpose(g)
    gtr = gnn.Graph(rpt, cit, None, None, False)
    dout = torch.randn((n, HD), dtype=torch.float32, device="cuda")
    gnn.gnn_projection(H, W, out=C)
    b_bwd = 2 * n * HD * 2 + 2 * n * HD * 4 + n * HD * 4 + 2 * n * HD * 4 + 4 * n * heads * 4 + 2 * idx
    timed = {"gatv2_backward": (
        lambda: gnn.gnn_gatv2_attn_bwd(g, gtr, C, None, a, heads, D, out, lse, dout, w["slope"]),
        b_bwd, "dl and da over CSR, dr over CSR^T, from the forward's out and lse (one projection: "
               "dC = dl + dr); timed apart, cold")}
    # the Graph Transformer backward on this power-law graph (8 heads x 32,
    # bf16 Q, K, V N(0,1) from the GT seeds): the edge-run schedule its mean
    # degree selects, hub rows of ~40K edges cut into 256-edge pieces
    gh, gd = 8, 32
    gq, gk, gv = (_dev(torch, synth_mod().normal_bf16((n, gh * gd), 1.0, s)) for s in (4, 5, 6))
    gout = torch.empty((n, gh * gd), dtype=torch.float32, device="cuda")
    glse = torch.empty((n, gh), dtype=torch.float32, device="cuda")
    gscale = 1.0 / float(np.sqrt(gd))
    gnn.gnn_gt_attn_fwd(g, gq, gk, gv, gh, gd, gscale, out=gout, lse=glse)
    gdout = torch.randn((n, gh * gd), dtype=torch.float32, device="cuda")
    b_gt = 3 * n * gh * gd * 2 + 2 * n * gh * gd * 4 + 3 * n * gh * gd * 4 + 2 * idx
    timed["gt_backward_rmat20"] = (
        lambda: gnn.gnn_gt_attn_bwd(g, gtr, gq, gk, gv, gh, gd, gscale, gout, glse, gdout),
        b_gt, "Graph Transformer backward on this graph (8 heads x 32, bf16 Q, K, V): dQ over CSR, "
              "dK and dV over CSR^T on 256-edge runs (hub rows cut and summed in edge order); timed "
              "apart, cold")
    cfg = {"workload": "c3_rmat20_gatv2", "graph": "R-MAT scale 20, edge factor 16, dedup + "
           "self-loops", "nodes": n, "edges": M, "heads": heads, "head_dim": D, "f_in": 256,
           "dtype": "bf16 H, W and C; fp32 softmax and accumulation; fp32 out",
           "layers": ["tcgen05 projection + fused GATv2 (score, online softmax, aggregate)"]}
    rows = _sample_by_edges(w["rowptr"], 40000)
    return Workload("c3_rmat20_gatv2", layers, [H], [out, lse], cfg, "bf16", oracle_step, rows,
                    extra={"proj_only": (proj_only, b_proj), "b_attn": b_attn, "timed": timed,
                           "unfused": (g, H, W, a, heads, D, w["slope"])})


def setup_c4(torch, gnn, w, tiles=None, packing=0):
    """GT attention on the clustered graph.  tiles = None: the CSR path;
    a number: the tile path at that fill threshold; "auto": the backend and
    threshold the adaptive selector picks, timed first, with the other path
    timed beside it."""
    g = gnn.graph_prepare(_dev(torch, w["rowptr"]), _dev(torch, w["colidx"]))
    Q, K, V = (_dev(torch, w[k]) for k in ("Q", "K", "V"))
    n = Q.shape[0]
    M = len(w["colidx"])
    heads, D = w["heads"], w["head_dim"]
    HD = heads * D
    out = torch.empty((n, HD), dtype=torch.float32, device="cuda")
    lse = torch.empty((n, heads), dtype=torch.float32, device="cuda")
    idx = 4 * (n + 1) + 4 * M
    bcomp = idx + 3 * n * HD * 2 + n * HD * 4 + n * heads * 4
    extra = {"selector": selector_report(torch, gnn, g, gnn.GNN_OP_GT, gnn.GNN_BF16, 0, heads, D)}
    sel = extra["selector"]
    both = tiles == "auto"
    if both:
        tiles = sel["fill_threshold"] if sel["backend"] == "tiles" else None
    bs = None
    if tiles is not None:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        bs = gnn.gnn_blocksparse_build(g, tiles, packing=packing)
        torch.cuda.synchronize()
        m = bs.meta
        extra["blocksparse"] = {"threshold": tiles, "packing": ["id", "count"][packing],
                                "build_ms": (time.perf_counter() - t0) * 1e3,
                                "listed_blocks": m.n_blocks, "kept_tiles": m.n_tiles_kept,
                                "tile_edges": m.nnz_tiles, "residual_edges": m.nnz_residual,
                                # S = Q K^T and O = P V over every listed block's 16 columns
                                "tile_mma_flop": 4.0 * 128 * D * 16 * m.n_blocks * heads}

    def gt_layer(use_bs):
        nm = "gt_tiles" if use_bs is not None else "gt_csr"
        return Layer(nm, lambda ins: gnn.gnn_gt_attn_fwd(g, ins[0], ins[1], ins[2], heads, D,
                                                         w["scale"], bs=use_bs, out=out, lse=lse),
                     M * HD, bcomp, "alu" if use_bs is None else "tensor")

    layers = [gt_layer(bs)]
    if both and bs is not None:
        layers.append(gt_layer(None))
    if bs is None or both:
        # backward of the attention (transpose built once here), from the
        # forward's out and lse, which every path leaves identical
        rpt, cit, _ = gnn.gnn_csr_transpose(g)
        gtr = gnn.Graph(rpt, cit, None, None, False)
        dout = torch.randn((n, HD), dtype=torch.float32, device="cuda")
        bwd_bytes = 3 * n * HD * 2 + 2 * n * HD * 4 + 3 * n * HD * 4 + 2 * (idx + 4 * M)
        extra["timed"] = {"gt_backward": (
            lambda: gnn.gnn_gt_attn_bwd(g, gtr, Q, K, V, heads, D, w["scale"], out, lse, dout),
            bwd_bytes, "dQ over CSR, dK and dV over CSR^T (Delta fused into the dQ pass), from "
                       "the forward's out and lse; timed apart, cold")}

    def oracle_step(rows):
        import oracle
        oracle.gt(w["rowptr"], w["colidx"], w["Q"], w["K"], w["V"], heads, D, w["scale"],
                  rows=rows)

    desc = ("fused GT attention, CSR path" if bs is None else
            f"GT attention: tcgen05 16x16 tiles (fill >= {tiles}) + CSR residual")
    cfg = {"workload": "c4_clustered_gt", "graph": "1024 clusters x 256 nodes, p=0.3, 1% of "
           "sources rewired, dedup + self-loops", "nodes": n, "edges": M, "heads": heads,
           "head_dim": D, "dtype": "bf16 Q, K, V; fp32 softmax and accumulation; fp32 out",
           "layers": [desc] + (["fused GT attention, CSR path (beside the selected one)"]
                               if len(layers) > 1 else [])}
    rows = _sample_by_edges(w["rowptr"], 400000)
    # with "auto" the selected layer comes first and the other is timed beside it
    return Workload("c4_clustered_gt", layers, [Q, K, V], [out, lse], cfg, "bf16", oracle_step,
                    rows, extra=extra)


def setup_c4_spmm(torch, gnn, w, tiles=None, packing=0):
    """GCN SpMM (norm BOTH) on the clustered graph of the GT workload with X
    bf16 [N, 256] N(0,1): the CSR edge-span kernel, or with tiles the
    tensor-core SpMM over the block-sparse layout plus the residual CSR."""
    g = gnn.graph_prepare(_dev(torch, w["rowptr"]), _dev(torch, w["colidx"]))
    n = len(w["rowptr"]) - 1
    M = len(w["colidx"])
    F = 256
    Xh = synth_mod().normal_bf16((n, F), 1.0, 44)
    X = _dev(torch, Xh)
    Y = torch.empty((n, F), dtype=torch.float32, device="cuda")
    idx = 4 * (n + 1) + 4 * M
    bcomp = idx + n * F * 2 + n * F * 4 + 8 * n
    extra = {}
    bs = None
    if tiles is not None:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        bs = gnn.gnn_blocksparse_build(g, tiles, packing=packing)
        torch.cuda.synchronize()
        m = bs.meta
        extra["blocksparse"] = {"threshold": tiles, "packing": ["id", "count"][packing],
                                "build_ms": (time.perf_counter() - t0) * 1e3,
                                "listed_blocks": m.n_blocks, "kept_tiles": m.n_tiles_kept,
                                "tile_edges": m.nnz_tiles, "residual_edges": m.nnz_residual,
                                # O += P X over every listed block's 16 columns
                                "tile_mma_flop": 2.0 * 128 * 16 * F * m.n_blocks}
        layers = [Layer("spmm_tiles", lambda ins: gnn.gnn_spmm_blocksparse(
            g, ins[0], bs, norm=gnn.GNN_NORM_BOTH, out=Y), M * F, bcomp, "tensor")]
    else:
        layers = [Layer("spmm", lambda ins: gnn.gnn_spmm(g, ins[0], norm=gnn.GNN_NORM_BOTH,
                                                         out=Y), M * F, bcomp)]

    def oracle_step(rows):
        import oracle
        oracle.spmm(w["rowptr"], w["colidx"], Xh, norm=oracle.NORM_BOTH, rows=rows)

    cfg = {"workload": "c4_clustered_spmm", "graph": "the GT workload's clustered graph: 1024 "
           "clusters x 256 nodes, p=0.3, 1% of sources rewired, dedup + self-loops",
           "nodes": n, "edges": M, "features": F, "x_dtype": "bf16",
           "layers": ["gcn_spmm, CSR edge spans" if bs is None else
                      f"gcn_spmm: tcgen05 16x16 tiles (fill >= {tiles}) + CSR residual"]}
    rows = _sample_by_edges(w["rowptr"], 2000000)
    return Workload("c4_clustered_spmm", layers, [X], [Y], cfg, "bf16", oracle_step, rows,
                    extra=extra)


def synth_mod():
    import synth
    return synth


def setup_c5(torch, gnn, w, mapping="auto", ordering="original"):
    rp, ci = _dev(torch, w["rowptr"]), _dev(torch, w["colidx"])
    X = _dev(torch, w["X"])
    n, F = X.shape
    M = len(w["colidx"])
    prep = {}
    if ordering != "original":
        kind = {"random": gnn.GNN_PERM_RANDOM, "degree": gnn.GNN_PERM_DEGREE,
                "rcm": gnn.GNN_PERM_RCM}[ordering]
        g0 = gnn.Graph(rp, ci, prepare=False)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        perm, inv = gnn.gnn_reorder_perm(g0, kind, 7)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        rp, ci, X = gnn.gnn_apply_perm(g0, perm, inv, X=X)
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        prep = {"order_ms": (t1 - t0) * 1e3, "relabel_ms": (t2 - t1) * 1e3}
        del g0, perm, inv
    g = gnn.graph_prepare(rp, ci)
    Y = torch.empty((n, F), dtype=torch.float32, device="cuda")
    mp = {"auto": gnn.GNN_MAP_AUTO, "feat": gnn.GNN_MAP_FEAT, "neigh": gnn.GNN_MAP_NEIGH}[mapping]
    idx = 4 * (n + 1) + 4 * M
    bcomp = idx + n * F * 2 + n * F * 4 + 8 * n
    layers = [Layer("spmm", lambda ins: gnn.gnn_spmm(g, ins[0], norm=gnn.GNN_NORM_BOTH,
                                                     mapping=mp, out=Y), M * F, bcomp)]

    def oracle_step(rows):
        import oracle
        oracle.spmm(w["rowptr"], w["colidx"], w["X"], norm=oracle.NORM_BOTH, rows=rows)

    cfg = {"workload": "c5_rmat22", "graph": "R-MAT scale 22, edge factor 16, dedup + "
           "self-loops", "nodes": n, "edges": M, "features": F, "x_dtype": "bf16",
           "ordering": ordering, "mapping": mapping, "layers": ["gcn_spmm"]}
    # ~16M edges x 256 features of single-core oracle work (~10 s)
    rows = _sample_by_edges(w["rowptr"], 16000000)
    extra = {"graph": g}
    if prep:
        extra["reorder_prep"] = prep
    return Workload("c5_rmat22", layers, [X], [Y], cfg, "bf16", oracle_step, rows, extra=extra)


SETUPS = {"c2_rmat17": setup_c2, "c3_rmat20_gatv2": setup_c3, "c4_clustered_gt": setup_c4,
          "c4_clustered_spmm": setup_c4_spmm,
          "c5_rmat22": setup_c5}


# ---------------------------------------------------------------- main

def max_over_ranks(torch, ms, world):
    """The slowest rank's time (all_reduce MAX over the process group, on its
    backend's device): the job is done when every rank is."""
    if world <= 1:
        return ms
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, steps, total_ms):
    """Whole-job throughput in G units/s: each rank processed units_per_rank
    a step for `steps` steps, and the job took the slowest rank's total_ms."""
    return world * units_per_rank * steps / (total_ms * 1e-3) / 1e9


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def with_feature_width(synth, w, args):
    """c2 with --features F: X regenerated as N(0, 1) fp32 [N, F] (same seed)."""
    if args.features and args.workload == "c2_rmat17":
        w["X"] = synth.normal_f32((len(w["rowptr"]) - 1, args.features), 1.0, synth.SEED_X)
    return w


def run_reference(args):
    import synth
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = synth.workload("c4_clustered_gt", features=False) if args.workload == "c4_clustered_spmm" \
        else with_feature_width(synth, synth.workload(args.workload), args)
    wl_meta = REF_META[args.workload](w)
    rows, ne, per_edge, fn = wl_meta
    for _ in range(args.warmup):
        fn(rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        fn(rows)
    dt = (time.perf_counter() - t) / args.steps
    v = ne * per_edge / dt / 1e9
    wname = args.workload
    if args.features and args.workload == "c2_rmat17" and args.features != 128:
        wname = f"c2_rmat17_f{args.features}"
    sample = f"{len(rows)} destination rows ({ne} edges) of {wname} per step"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wname, "sample": sample},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "cpu_model": host_cpu()[0], "nproc": host_cpu()[1],
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _ref_c2(w):
    import oracle
    rp, ci, X = w["rowptr"], w["colidx"], w["X"]
    rows = np.arange(0, len(rp) - 1, 16, dtype=np.int32)
    ne = int(np.sum(rp[rows + 1] - rp[rows]))

    def fn(r):
        oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH, rows=r)
        oracle.segment_reduce(oracle.OP_SUM, rp, ci, X, rows=r)
        oracle.segment_reduce(oracle.OP_MEAN, rp, ci, X, rows=r)
        oracle.segment_reduce(oracle.OP_MAX, rp, ci, X, rows=r)
    return rows, ne, 4 * X.shape[1], fn


def _ref_c3(w):
    import oracle
    rows, ne = _sample_by_edges(w["rowptr"], 4000)
    HD = w["heads"] * w["head_dim"]

    def fn(r):
        oracle.gatv2(w["rowptr"], w["colidx"], w["H"], w["W"], w["a"], w["heads"], w["head_dim"],
                     w["slope"], rows=r)
    return rows, ne, HD, fn


def _ref_c4(w):
    import oracle
    rows, ne = _sample_by_edges(w["rowptr"], 100000)
    HD = w["heads"] * w["head_dim"]

    def fn(r):
        oracle.gt(w["rowptr"], w["colidx"], w["Q"], w["K"], w["V"], w["heads"], w["head_dim"],
                  w["scale"], rows=r)
    return rows, ne, HD, fn


def _ref_c5(w):
    import oracle
    rows, ne = _sample_by_edges(w["rowptr"], 1000000)

    def fn(r):
        oracle.spmm(w["rowptr"], w["colidx"], w["X"], norm=oracle.NORM_BOTH, rows=r)
    return rows, ne, w["X"].shape[1], fn


def _ref_c4_spmm(w):
    import oracle
    import synth
    rp, ci = w["rowptr"], w["colidx"]
    X = synth.normal_bf16((len(rp) - 1, 256), 1.0, 44)
    rows, ne = _sample_by_edges(rp, 400000)

    def fn(r):
        oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH, rows=r)
    return rows, ne, 256, fn


REF_META = {"c2_rmat17": _ref_c2, "c3_rmat20_gatv2": _ref_c3, "c4_clustered_gt": _ref_c4,
            "c5_rmat22": _ref_c5, "c4_clustered_spmm": _ref_c4_spmm}


def _ev(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def time_cold(torch, fn, steps, flush, stream):
    """fn() K times, each after an L2 flush (outside the events); per-call ms."""
    evs = [_ev(torch) for _ in range(steps)]
    for k, (e0, e1) in enumerate(evs):
        flush.fill_(float(k))
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def time_e2e_sequential(torch, W, steps, flush, stream, ins_h, outs_h):
    """One step at a time through the public API: copy the inputs in from
    pinned host memory, run the layers, read the results back; one untimed
    step first, then `steps` steps, each in its own events (L2 flushed before
    each, outside the events).  Per-step ms."""
    ins_d = [torch.empty_like(x, device="cuda") for x in ins_h]

    def one():
        for xd, xh in zip(ins_d, ins_h):
            xd.copy_(xh, non_blocking=True)
        W.step(ins=ins_d)
        for oh, od in zip(outs_h[0], W.outputs):
            oh.copy_(od, non_blocking=True)

    one()
    ms = time_cold(torch, one, steps, flush, stream)
    del ins_d
    return ms


def time_e2e_pipelined(torch, W, steps, warmup, stream, ins_h, outs_h, runs=3):
    """Steps as a serving loop runs them: three streams (copy in, compute,
    copy out) and two buffers of each kind, so that step k+1's input copy and
    step k-1's read-back overlap step k's kernels.  Every step still copies
    its own inputs from pinned host memory and reads its own results back
    into pinned host memory inside the timed region.  The step's output
    tensors are pointed (Tensor.set_) at one of two device buffers before
    each step, so the kernels write straight into the buffer whose previous
    read-back has finished, with no staging copy.  `warmup` untimed steps,
    then `runs` timed runs of `steps` steps each (the host link is shared
    with the rest of the machine, so a single run can catch a stall); returns
    each run's ms per step."""
    ins_d = [[torch.empty_like(x, device="cuda") for x in ins_h] for _ in range(2)]
    outs_d = [[torch.empty_like(o) for o in W.outputs] for _ in range(2)]
    keep = [o.detach() for o in W.outputs]  # the outputs' own storage, restored after
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def run(K, timed):
        ev_in = [torch.cuda.Event() for _ in range(K)]
        ev_c = [torch.cuda.Event() for _ in range(K)]
        ev_out = [torch.cuda.Event() for _ in range(K)]
        t0, t1 = _ev(torch)
        torch.cuda.synchronize()
        t0.record(stream)
        s_in.wait_event(t0)
        s_out.wait_event(t0)
        for k in range(K):
            b = k & 1
            with torch.cuda.stream(s_in):
                if k >= 2:  # input buffer b is free once step k-2's kernels have read it
                    s_in.wait_event(ev_c[k - 2])
                for xd, xh in zip(ins_d[b], ins_h):
                    xd.copy_(xh, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if k >= 2:  # output buffer b is free once step k-2's read-back is done
                stream.wait_event(ev_out[k - 2])
            for o, od in zip(W.outputs, outs_d[b]):
                o.set_(od)
            W.step(ins=ins_d[b])
            ev_c[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[k])
                for oh, od in zip(outs_h[b], outs_d[b]):
                    oh.copy_(od, non_blocking=True)
                ev_out[k].record(s_out)
        stream.wait_event(ev_out[K - 1])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / K if timed else None

    try:
        run(max(2, warmup), False)
        ms = [run(steps, True) for _ in range(runs)]
    finally:
        torch.cuda.synchronize()
        for o, k0 in zip(W.outputs, keep):
            o.set_(k0)
    del ins_d, outs_d
    return ms


def time_warm(torch, fn, steps, stream):
    """fn() K times back to back (the caches keep what the last call left)."""
    fn()
    evs = [_ev(torch) for _ in range(steps)]
    for e0, e1 in evs:
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def time_warm_graph(torch, fn, steps, stream, reps=20):
    """fn() `reps` times back to back captured in one CUDA graph, replayed
    `steps` times: the warm per-call time without per-launch host overhead
    (the layers of the scale-17 workload are tens of microseconds).  Returns
    (per-call ms list, None) or (None, the capture error)."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        evs = [_ev(torch) for _ in range(steps)]
        for e0, e1 in evs:
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        out = [e0.elapsed_time(e1) / reps for e0, e1 in evs]
        del graph
        return out, None
    except Exception as e:  # reported in the line, the cold and warm figures stand
        torch.cuda.synchronize()
        return None, f"{type(e).__name__}: {str(e)[:160]}"


def summary(ms):
    return {"ms_median": float(np.median(ms)), "ms_min": float(np.min(ms)),
            "ms_mean": float(np.mean(ms))}


def time_layers(torch, W, steps, flush, stream):
    """K steps of W; an L2 flush precedes every layer of every step, outside
    the events.  Returns (per-step ms = sum of its layers, per-layer ms lists)."""
    names = [L.name for L in W.layers]
    ev = [{k: _ev(torch) for k in names} for _ in range(steps)]
    for k in range(steps):
        for L in W.layers:
            flush.fill_(float(k))
            ev[k][L.name][0].record(stream)
            L.fn(W.inputs)
            ev[k][L.name][1].record(stream)
    torch.cuda.synchronize()
    per = {nm: [e[nm][0].elapsed_time(e[nm][1]) for e in ev] for nm in names}
    step_ms = [sum(per[nm][k] for nm in names) for k in range(steps)]
    return step_ms, per


def layer_report(torch, W, L, cold_ms, warm_ms, hbm):
    """One layer's numbers: cold median / min / mean, warm median, its rate
    and its compulsory-byte fraction of the HBM peak (from the cold mean)."""
    c = summary(cold_ms)
    t = c["ms_mean"]
    gbs = L.bcomp / (t * 1e-3) / 1e9
    r = {"ms": t, **c, "warm_ms_median": float(np.median(warm_ms)),
         "gedge_feat_s": L.units / (t * 1e-3) / 1e9, "bcomp_bytes": L.bcomp, "hbm_gbs": gbs,
         "frac": gbs / hbm, "frac_of_8tbs": gbs / NOMINAL_HBM_GBS, "bound": L.bound}
    tr, _ = recorded_traffic(W.name, L.name)
    if tr is not None:
        r["dram_bytes_ncu"] = tr
        r["dram_over_bcomp"] = tr / L.bcomp
    return r


def timed_extras(torch, W, steps, flush, stream, hbm, layers):
    """The workload's side measurements, each cold (flush before every call)."""
    extra = {}
    if "selector" in W.extra:
        extra["selector"] = W.extra["selector"]
    if "reorder_prep" in W.extra:
        extra["reorder_prep"] = W.extra["reorder_prep"]
    if "blocksparse" in W.extra:
        bsx = dict(W.extra["blocksparse"])
        bsx["tile_mma_tflops"] = bsx["tile_mma_flop"] / (layers[W.layers[0].name]["ms"] * 1e-3) / 1e12
        extra["blocksparse"] = bsx
    for tname, spec in W.extra.get("timed", {}).items():
        fn, tbytes, tnote = spec[:3]
        tunits = spec[3] if len(spec) > 3 else None
        fn()
        c = summary(time_cold(torch, fn, steps, flush, stream))
        t = c["ms_mean"]
        e = {"ms": t, **c, "note": tnote}
        if tbytes:
            e.update(bytes=tbytes, hbm_gbs=tbytes / (t * 1e-3) / 1e9,
                     frac=tbytes / (t * 1e-3) / 1e9 / hbm)
        if tunits:
            e["gedge_feat_s"] = tunits / (t * 1e-3) / 1e9
        extra[tname] = e
    if "proj_only" in W.extra:
        fn, b_proj = W.extra["proj_only"]
        c = summary(time_cold(torch, fn, steps, flush, stream))
        pms = c["ms_median"]
        gat = layers["gatv2_fwd"]["ms_median"]
        extra["projection_alone"] = {"ms": pms, **c, "bytes": b_proj,
                                     "hbm_gbs": b_proj / (pms * 1e-3) / 1e9,
                                     "frac": b_proj / (pms * 1e-3) / 1e9 / hbm,
                                     "tflops": 2 * W.inputs[0].shape[0] * 256 * 256 / (pms * 1e-3) / 1e12}
        att_ms = max(gat - pms, 1e-6)
        extra["attention_by_difference"] = {
            "ms": att_ms, "note": "layer median minus projection median", "bytes": W.extra["b_attn"],
            "hbm_gbs": W.extra["b_attn"] / (att_ms * 1e-3) / 1e9,
            "frac": W.extra["b_attn"] / (att_ms * 1e-3) / 1e9 / hbm}
    return extra


def unfused_gatv2_peak(torch, gnn, args_tuple):
    """Edge-materialising comparator (plain PyTorch ops): the per-edge
    scores, weights and messages of an unfused GATv2 layer are written to
    device memory, as message-passing frameworks do.  Returns (ms, peak
    bytes above the inputs)."""
    g, H, W, a, heads, D, slope = args_tuple
    rp = g.rowptr.long()
    ci = g.colidx.long()
    n = H.shape[0]
    dst = torch.repeat_interleave(torch.arange(n, device="cuda"), rp[1:] - rp[:-1])
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    C = (H.float() @ W.float()).view(n, heads, D)
    x = C[dst] + C[ci]                                        # [M, heads, D]
    e = (torch.nn.functional.leaky_relu(x, slope) * a.view(1, heads, D)).sum(-1)  # [M, heads]
    del x
    m = torch.full((n, heads), -float("inf"), device="cuda").index_reduce_(0, dst, e, "amax")
    p = torch.exp(e - m[dst])
    s = torch.zeros((n, heads), device="cuda").index_add_(0, dst, p)
    alpha = p / s[dst]
    msg = alpha.unsqueeze(-1) * C[ci]                          # [M, heads, D]
    out = torch.zeros((n, heads, D), device="cuda").index_add_(0, dst, msg)
    t1.record()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    del C, e, m, p, s, alpha, msg, out
    torch.cuda.empty_cache()
    return t0.elapsed_time(t1), peak


def load_workload(synth, name, args):
    if name == "c4_clustered_spmm":
        return synth.workload("c4_clustered_gt", features=False)
    if args.scale is not None:
        return with_feature_width(synth, rescaled(synth, name, args.scale), args)
    return with_feature_width(synth, synth.workload(name), args)


def rescaled(synth, name, scale):
    """An R-MAT workload at another scale (same edge factor, a,b,c,d, seeds
    and feature recipe): the small cases that ncu captures are sized on."""
    if name not in ("c2_rmat17", "c3_rmat20_gatv2", "c5_rmat22"):
        raise SystemExit(f"--scale applies to the R-MAT workloads, not {name}")
    rp, ci = synth.rmat(scale, 16, *synth.RMAT_ABC)
    n = 1 << scale
    w = {"name": name, "rowptr": rp, "colidx": ci, "n": n}
    if name == "c2_rmat17":
        w["X"] = synth.normal_f32((n, 128), 1.0, synth.SEED_X)
    elif name == "c3_rmat20_gatv2":
        w["H"] = synth.normal_bf16((n, 256), 1.0, synth.SEED_X)
        w["W"] = synth.normal_bf16((256, 256), 1.0 / 256, synth.SEED_W)
        w["a"] = synth.normal_f32((4, 64), 1.0 / 64, synth.SEED_A)
        w.update(heads=4, head_dim=64, slope=0.2)
    else:
        w["X"] = synth.normal_bf16((n, 256), 1.0, synth.SEED_X)
    return w


def setup_workload(torch, gnn, w, name, args, family=False):
    if name == "c5_rmat22":
        return setup_c5(torch, gnn, w, args.mapping, args.ordering)
    pk = {"id": 0, "count": 1}[args.packing]
    if name == "c4_clustered_gt":
        return setup_c4(torch, gnn, w, "auto" if family else args.tiles, 0 if family else pk)
    if name == "c4_clustered_spmm":
        return setup_c4_spmm(torch, gnn, w, args.tiles, pk)
    return SETUPS[name](torch, gnn, w)


def measure(torch, gnn, W, args, flush, stream, hbm, base_bytes):
    """Warm-up, then K cold steps (flush before every layer) and K warm calls
    per layer.  Returns (per-step ms, {layer: report}, launches in the cold
    steps, peak device memory of the warm-up above base_bytes, the memory
    held before the workload was set up)."""
    torch.cuda.reset_peak_memory_stats()
    for _ in range(args.warmup):
        W.step()
    torch.cuda.synchronize()
    peak_mem = torch.cuda.max_memory_allocated() - base_bytes
    launches0 = gnn.launch_count()
    step_ms, per = time_layers(torch, W, args.steps, flush, stream)
    launches = gnn.launch_count() - launches0
    layers = {}
    for L in W.layers:
        warm = time_warm(torch, lambda: L.fn(W.inputs), args.steps, stream)
        layers[L.name] = layer_report(torch, W, L, per[L.name], warm, hbm)
        if W.name == "c2_rmat17":
            g_ms, g_err = time_warm_graph(torch, lambda: L.fn(W.inputs), args.steps, stream)
            if g_ms is not None:
                layers[L.name]["warm_graph_ms_median"] = float(np.median(g_ms))
            else:
                layers[L.name]["warm_graph_error"] = g_err
    return step_ms, layers, launches, peak_mem


def run_family(torch, gnn, synth, name, args, flush, stream, hbm):
    """One family of the default run, on its own graph: its layers cold and
    warm, its side measurements, then its device memory is released."""
    base = torch.cuda.memory_allocated()
    w = load_workload(synth, name, args)
    W = setup_workload(torch, gnn, w, name, args, family=True)
    _, layers, _, peak_mem = measure(torch, gnn, W, args, flush, stream, hbm, base)
    rep = {"config": W.config, "layers": layers, "peak_memory_bytes": peak_mem}
    rep.update(timed_extras(torch, W, args.steps, flush, stream, hbm, layers))
    if name == "c3_rmat20_gatv2" and not args.no_comparator:
        ums, upeak = unfused_gatv2_peak(torch, gnn, W.extra["unfused"])
        rep["unfused_torch_comparator"] = {"ms": ums, "peak_bytes_above_inputs": upeak,
                                           "fused_peak_bytes": peak_mem,
                                           "peak_memory_ratio": upeak / max(peak_mem, 1),
                                           "speedup": ums / layers["gatv2_fwd"]["ms_median"]}
    del W, w
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rep


def run_study(torch, gnn, synth, args, flush, stream, hbm):
    """The ordering x mapping study of IO-aware GNN layers, Section 4.1 /
    App. E.1, on R-MAT scale 22: GCN SpMM under the AUTO (edge spans),
    feature-parallel and neighbour-parallel mappings after each vertex
    ordering; s = t_original / t_reordered per mapping, and
    delta_s = s_neighbour - s_feature per ordering.  Each cell is the cold
    median over K calls."""
    w = synth.workload("c5_rmat22")
    cells, prep = {}, {}
    for ordering in ("original", "random", "degree", "rcm"):
        W = setup_c5(torch, gnn, w, "auto", ordering)
        L = W.layers[0]
        prep[ordering] = W.extra.get("reorder_prep", {})
        g, X, Y = W.extra["graph"], W.inputs[0], W.outputs[0]
        for mname, mp in (("auto", gnn.GNN_MAP_AUTO), ("feat", gnn.GNN_MAP_FEAT),
                          ("neigh", gnn.GNN_MAP_NEIGH)):
            fn = (lambda mp=mp: gnn.gnn_spmm(g, X, norm=gnn.GNN_NORM_BOTH, mapping=mp, out=Y))
            for _ in range(args.warmup):
                fn()
            c = summary(time_cold(torch, fn, args.steps, flush, stream))
            gbs = L.bcomp / (c["ms_median"] * 1e-3) / 1e9
            cells[f"{ordering}/{mname}"] = {**c, "gedge_feat_s": L.units / (c["ms_median"] * 1e-3) / 1e9,
                                           "frac": gbs / hbm}
        del W, g, X, Y
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    t = {k: v["ms_median"] for k, v in cells.items()}
    s = {f"{o}/{m}": t[f"original/{m}"] / t[f"{o}/{m}"]
         for o in ("random", "degree", "rcm") for m in ("auto", "feat", "neigh")}
    ds = {o: s[f"{o}/neigh"] - s[f"{o}/feat"] for o in ("random", "degree", "rcm")}
    return {"study": "c5_rmat22 orderings x mappings (GCN SpMM, bf16 X [N,256], fp32 out)",
            "cells": cells, "s": s, "delta_s_neigh_minus_feat": ds, "reorder_prep_ms": prep,
            "steps": args.steps, "l2": "512 MB flush before every timed call (cold)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(SETUPS),
                    help="run one workload alone (default: the c5_rmat22 SpMM step plus the "
                         "c2, c3 and c4 families)")
    ap.add_argument("--features", type=int, default=None,
                    help="c2_rmat17 only: feature width F (fp32, a multiple of 4; default 128)")
    ap.add_argument("--mapping", default="auto", choices=["auto", "feat", "neigh"],
                    help="SpMM kernel mapping (c5_rmat22)")
    ap.add_argument("--ordering", default="original",
                    choices=["original", "random", "degree", "rcm"],
                    help="vertex ordering applied before timing (c5_rmat22; prep timed apart)")
    ap.add_argument("--tiles", type=float, default=None,
                    help="c4 workloads: tensor-core tile path at this fill threshold")
    ap.add_argument("--scale", type=int, default=None,
                    help="R-MAT workloads at this scale instead of their own (small cases "
                         "for profiling; the line's config names the scale)")
    ap.add_argument("--packing", default="id", choices=["id", "count"],
                    help="c4 tile paths: column order inside a row group (id, or descending "
                         "edge count)")
    ap.add_argument("--study", default=None, choices=["orderings"],
                    help="orderings: the R-MAT scale 22 SpMM under every vertex ordering and "
                         "kernel mapping (one JSON line; no headline step)")
    ap.add_argument("--no-families", action="store_true",
                    help="default run: the headline step only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-comparator", action="store_true",
                    help="skip the unfused GATv2 comparator (c3_rmat20_gatv2)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    suite = args.workload is None
    if suite and args.scale is not None:
        raise SystemExit("--scale needs --workload (one R-MAT workload)")
    if suite:
        args.workload = HEADLINE
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
    hbm, bf16_tf, peak_kind = measured_peaks()
    if args.study:
        stream = torch.cuda.current_stream()
        flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
        clocks = ClockSampler(local)
        clocks.start()
        rep = run_study(torch, gnn, synth, args, flush, stream, hbm)
        rep["clocks"] = clocks.stop()
        if rank == 0:
            print(json.dumps(rep), flush=True)
        return

    stream = torch.cuda.current_stream()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    base = torch.cuda.memory_allocated()
    w = load_workload(synth, args.workload, args)
    W = setup_workload(torch, gnn, w, args.workload, args)
    if args.scale is not None:
        # a rescaled R-MAT graph: its own name, so no recorded figure of the
        # full workload is attached to it
        W.name = f"{W.name}_at_scale{args.scale}"
        W.config["workload"] = W.name
        W.config["graph"] = f"R-MAT scale {args.scale}, edge factor 16, dedup + self-loops"

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    step_ms, layers, launches, peak_mem = measure(torch, gnn, W, args, flush, stream, hbm, base)
    barrier()
    total_ms = max_over_ranks(torch, float(np.sum(step_ms)), world)
    ms = total_ms / args.steps
    units = sum(L.units for L in W.layers)
    value = job_rate(world, units, args.steps, total_ms)
    extra = timed_extras(torch, W, args.steps, flush, stream, hbm, layers)
    if args.workload == "c3_rmat20_gatv2" and not args.no_comparator:
        ums, upeak = unfused_gatv2_peak(torch, gnn, W.extra["unfused"])
        extra["unfused_torch_comparator"] = {"ms": ums, "peak_bytes_above_inputs": upeak,
                                             "fused_peak_bytes": peak_mem,
                                             "peak_memory_ratio": upeak / max(peak_mem, 1),
                                             "speedup": ums / layers["gatv2_fwd"]["ms_median"]}

    dom = max(W.layers, key=lambda L: layers[L.name]["ms"])
    d = layers[dom.name]
    traffic, sha = recorded_traffic(W.name, dom.name)
    roofline = {"bound": "hbm", "kernel": dom.name, "achieved": d["hbm_gbs"], "peak": hbm,
                "unit": "GB/s", "frac": d["hbm_gbs"] / hbm, "peak_kind": peak_kind,
                "frac_of_8tbs": d["hbm_gbs"] / NOMINAL_HBM_GBS, "traffic": traffic,
                "traffic_sources_sha16": sha, "bcomp_bytes": dom.bcomp,
                "duration": "mean of the K cold launches (CUDA events, launching stream)"}
    if dom.bound == "alu":
        roofline["note"] = ("kernel is FP32-ALU heavy; frac is its compulsory-byte rate "
                            "against the HBM peak")
    elif dom.bound == "tensor":
        roofline["note"] = ("tensor-core tiles; frac is the compulsory-byte rate against the "
                            "HBM peak, the tile MMA rate is in extra.blocksparse")

    e2e = None
    if not args.no_e2e:
        ins_h = [x.cpu().pin_memory() for x in W.inputs]
        outs_h = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in W.outputs]
                  for _ in range(2)]
        k_e2e = max(4, args.steps // 4)
        pipe = time_e2e_pipelined(torch, W, k_e2e, args.warmup, stream, ins_h, outs_h, runs=5)
        pipe_ms = max_over_ranks(torch, float(np.median(pipe)), world)
        seq = time_e2e_sequential(torch, W, max(3, args.steps // 4), flush, stream, ins_h, outs_h)
        seq_ms = max_over_ranks(torch, float(np.median(seq)), world)
        e2e = {"value": job_rate(world, units, 1, pipe_ms), "unit": UNIT,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in ins_h),
               "d2h_bytes_per_step": sum(o.numel() * o.element_size() for o in outs_h[0]),
               "ms_per_step": pipe_ms, "steps": k_e2e,
               "runs_ms_per_step": [round(x, 4) for x in pipe],
               "schedule": "pipelined: copy-in, compute and read-back streams, two buffers "
                           "each; every step's copies inside the timed run; median of "
                           f"{len(pipe)} runs of {k_e2e} steps",
               "sequential": {"value": job_rate(world, units, 1, seq_ms),
                              "ms_per_step_median": seq_ms,
                              "ms_per_step_min": float(np.min(seq)),
                              "ms_per_step_mean": float(np.mean(seq))}}
        del ins_h, outs_h

    families = {}
    if suite and not args.no_families:
        oracle_w, oracle_W = w, W
        for name in FAMILIES:
            families[name] = run_family(torch, gnn, synth, name, args, flush, stream, hbm)
        w, W = oracle_w, oracle_W
    clk = clocks.stop()

    cfg = dict(W.config)
    cfg["l2"] = "512 MB flush write before every timed layer (cold); warm = back to back"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": W.dtype, "data": "synthetic",
            "config": cfg, "roofline": roofline, "layers": layers, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clk,
            "peak_memory_bytes": peak_mem}
    if families:
        line["families"] = families
    if extra:
        line["extra"] = extra

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, ne = W.sample_rows
        t = time.perf_counter()
        W.oracle_step(rows)
        dt = time.perf_counter() - t
        per_edge = units / max(len(w["colidx"]), 1)
        model, ncpu = host_cpu()
        line["cpu_baseline"] = {"value": ne * per_edge / dt / 1e9, "unit": UNIT, "cores": 1,
                                "kind": "oracle", "cpu_model": model, "nproc": ncpu,
                                "sample": f"{len(rows)} destination rows ({ne} edges) of "
                                          f"{args.workload}, one step, {dt:.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
