"""Seeded synthetic inputs shared by the CUDA library's tests/benchmarks and
the CPU oracle's tests.

Holds no arithmetic of the aggregation method: it draws random numbers
(SplitMix64, counter based) and lays graphs out in the CSR input format
(rows = destination nodes, columns = source nodes, ascending within each row,
duplicates removed, one self-loop per node).

The five workload recipes mirror the shapes, sizes, value distributions and
degree structure of the workloads of "On efficient scaling of GNNs via
IO-aware layer implementations" (Section 4 setup, Appendix C dataset table),
which are public datasets not available here; synthetic graphs stand in for
them.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# stream ids (one per kind of draw) and seeds per input
SEED_GRAPH, SEED_X, SEED_W, SEED_A, SEED_Q, SEED_K, SEED_V, SEED_PERM = 0, 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            i32p = ctypes.POINTER(ctypes.c_int32)
            i32pp = ctypes.POINTER(i32p)
            lib.synth_er.restype = ctypes.c_int64
            lib.synth_er.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, i32p, i32pp]
            lib.synth_rmat.restype = ctypes.c_int64
            lib.synth_rmat.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_double, ctypes.c_uint64,
                                       i32p, i32pp]
            lib.synth_clustered.restype = ctypes.c_int64
            lib.synth_clustered.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_uint64, i32p, i32pp]
            lib.synth_take.argtypes = [i32p, i32p, ctypes.c_int64]
            lib.synth_uniform_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_normal_f32.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,
                                             ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_splitmix64.restype = ctypes.c_uint64
            lib.synth_splitmix64.argtypes = [ctypes.c_uint64]
            lib.synth_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _finish(n: int, rowptr: np.ndarray, colp, nnz: int):
    if nnz < 0:
        raise MemoryError("synth: out of host memory")
    colidx = np.empty(nnz, dtype=np.int32)
    _load().synth_take(_i32p(colidx), colp, nnz)
    return rowptr, colidx


def er(n: int, m: int, seed: int = SEED_GRAPH):
    """Erdos-Renyi G(n, m) directed, plus one self-loop per node."""
    lib = _load()
    rowptr = np.empty(n + 1, dtype=np.int32)
    colp = ctypes.POINTER(ctypes.c_int32)()
    nnz = lib.synth_er(n, m, seed, _i32p(rowptr), ctypes.byref(colp))
    return _finish(n, rowptr, colp, nnz)


def rmat(scale: int, edge_factor: int = 16, a: float = 0.57, b: float = 0.19,
         c: float = 0.19, seed: int = SEED_GRAPH):
    """R-MAT power-law graph, duplicates and generated self-loops removed,
    one self-loop per node added."""
    lib = _load()
    n = 1 << scale
    rowptr = np.empty(n + 1, dtype=np.int32)
    colp = ctypes.POINTER(ctypes.c_int32)()
    nnz = lib.synth_rmat(scale, edge_factor, a, b, c, seed, _i32p(rowptr), ctypes.byref(colp))
    return _finish(n, rowptr, colp, nnz)


def clustered(n_clusters: int = 1024, cluster_size: int = 256, p: float = 0.3,
              rewire: float = 0.01, seed: int = SEED_GRAPH):
    """Locally dense clustered graph (intra-cluster probability p, a fraction
    `rewire` of edges given a source outside the cluster), plus self-loops."""
    lib = _load()
    n = n_clusters * cluster_size
    rowptr = np.empty(n + 1, dtype=np.int32)
    colp = ctypes.POINTER(ctypes.c_int32)()
    nnz = lib.synth_clustered(n_clusters, cluster_size, p, rewire, seed, _i32p(rowptr),
                              ctypes.byref(colp))
    return _finish(n, rowptr, colp, nnz)


def uniform_f32(shape, lo: float, hi: float, seed: int, stream: int = 0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_uniform_f32(out.ctypes.data, out.size, lo, hi, seed, stream)
    return out


def normal_f32(shape, var: float, seed: int, stream: int = 0) -> np.ndarray:
    """N(0, var) (var is the variance), fp32."""
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(out.ctypes.data, out.size, 0.0, math.sqrt(var), seed, stream)
    return out


def normal_bf16(shape, var: float, seed: int, stream: int = 0) -> np.ndarray:
    """N(0, var) rounded to bf16 (round to nearest even); returned as the raw
    16-bit patterns in a uint16 array."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(out.ctypes.data, out.size, 0.0, math.sqrt(var), seed, stream)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def splitmix64(x: int) -> int:
    return int(_load().synth_splitmix64(x))


def threads() -> int:
    return int(_load().synth_num_threads())


# ---------------------------------------------------------------------------
# workload recipes
# ---------------------------------------------------------------------------

RMAT_ABC = (0.57, 0.19, 0.19)

WORKLOADS = {
    "c1_er1k": "Erdos-Renyi N=1024, 8192 edges + self-loops; X fp32 U[-1,1] [1024,32]; "
               "W fp32 [32,32] N(0,1/32); a [1,32] N(0,1/32); LeakyReLU slope 0.2",
    "c2_rmat17": "R-MAT scale 17, edge factor 16 (a,b,c,d=.57,.19,.19,.05); X fp32 N(0,1) [N,128]",
    "c3_rmat20_gatv2": "R-MAT scale 20, edge factor 16; H bf16 N(0,1) [N,256]; W bf16 [256,256] "
                       "N(0,1/256); a fp32 [4,64] N(0,1/64); 4 heads x 64",
    "c4_clustered_gt": "clustered 1024 clusters x 256 nodes, p=0.3, 1% rewired; Q,K,V bf16 N(0,1) "
                       "[N,8x32]; scale 1/sqrt(32)",
    "c5_rmat22": "R-MAT scale 22, edge factor 16; X bf16 N(0,1) [N,256]; GCN normalisation",
}


def workload(name: str, features: bool = True) -> dict:
    """Generate one workload.  Returns a dict of numpy arrays and scalars."""
    w: dict = {"name": name}
    if name == "c1_er1k":
        rp, ci = er(1024, 8192)
        w.update(rowptr=rp, colidx=ci, n=1024)
        if features:
            w["X"] = uniform_f32((1024, 32), -1.0, 1.0, SEED_X)
            w["W"] = normal_f32((32, 32), 1.0 / 32, SEED_W)
            w["a"] = normal_f32((1, 32), 1.0 / 32, SEED_A)
        w.update(heads=1, head_dim=32, slope=0.2)
    elif name == "c2_rmat17":
        rp, ci = rmat(17, 16, *RMAT_ABC)
        n = 1 << 17
        w.update(rowptr=rp, colidx=ci, n=n)
        if features:
            w["X"] = normal_f32((n, 128), 1.0, SEED_X)
    elif name == "c3_rmat20_gatv2":
        rp, ci = rmat(20, 16, *RMAT_ABC)
        n = 1 << 20
        w.update(rowptr=rp, colidx=ci, n=n)
        if features:
            w["H"] = normal_bf16((n, 256), 1.0, SEED_X)
            w["W"] = normal_bf16((256, 256), 1.0 / 256, SEED_W)
            w["a"] = normal_f32((4, 64), 1.0 / 64, SEED_A)
        w.update(heads=4, head_dim=64, slope=0.2)
    elif name == "c4_clustered_gt":
        rp, ci = clustered(1024, 256, 0.3, 0.01)
        n = 1024 * 256
        w.update(rowptr=rp, colidx=ci, n=n)
        if features:
            w["Q"] = normal_bf16((n, 256), 1.0, SEED_Q)
            w["K"] = normal_bf16((n, 256), 1.0, SEED_K)
            w["V"] = normal_bf16((n, 256), 1.0, SEED_V)
        w.update(heads=8, head_dim=32, scale=1.0 / math.sqrt(32.0))
    elif name == "c5_rmat22":
        rp, ci = rmat(22, 16, *RMAT_ABC)
        n = 1 << 22
        w.update(rowptr=rp, colidx=ci, n=n)
        if features:
            w["X"] = normal_bf16((n, 256), 1.0, SEED_X)
    else:
        raise KeyError(name)
    return w
