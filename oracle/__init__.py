"""CPU oracle (plain C, single thread, fp64 accumulation) -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline /
reference leg may import this package.  The CUDA library and its Python
binding never import it, and it shares no code with them.

Each wrapper takes numpy arrays (CSR by destination: rowptr int32 [N+1],
colidx int32 [M]; features fp32, or bf16 as raw uint16 bit patterns) and
returns numpy arrays in fp64.  ``rows`` selects a subset of destination rows
(the oracle then computes only those rows, which is how full-size workloads
are checked on sampled outputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NORM_NONE, NORM_LEFT, NORM_RIGHT, NORM_BOTH = 0, 1, 2, 3
OP_SUM, OP_MEAN, OP_MAX, OP_MIN = 0, 1, 2, 3

_VP = ctypes.c_void_p


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-shared", "-fPIC",
                               "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            i32, i64, dbl, flt = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_float
            lib.orc_degrees.argtypes = [i32, i32, _VP, _VP, _VP, _VP]
            lib.orc_spmm.argtypes = [i32, i32, _VP, _VP, _VP, ctypes.c_int, _VP, ctypes.c_int,
                                     i32, _VP, i32, _VP]
            lib.orc_segment_reduce.argtypes = [ctypes.c_int, i32, _VP, _VP, _VP, ctypes.c_int,
                                               i32, _VP, i32, _VP, _VP]
            lib.orc_reduce_ext_backward.argtypes = [i32, i32, i32, _VP, _VP, _VP]
            lib.orc_csr_transpose.argtypes = [i32, i32, _VP, _VP, _VP, _VP, _VP, _VP]
            lib.orc_gt_backward.argtypes = [i32, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, i32, i32, dbl,
                                            _VP, _VP, _VP, _VP]
            lib.orc_degree_stats.argtypes = [i32, _VP, _VP]
            lib.orc_gatv2_backward.argtypes = [i32, _VP, _VP, _VP, _VP, ctypes.c_int, _VP, i32, i32,
                                               dbl, _VP, _VP, _VP, _VP]
            lib.orc_gatv2.argtypes = [i32, _VP, _VP, _VP, ctypes.c_int, i32, _VP, _VP, _VP,
                                      i32, i32, dbl, _VP, i32, _VP, _VP, _VP]
            lib.orc_gatv2_ex.argtypes = [i32, _VP, _VP, _VP, ctypes.c_int, i32, _VP, _VP, _VP,
                                         i32, i32, dbl, _VP, i32, ctypes.c_int, _VP, _VP, _VP]
            lib.orc_gt.argtypes = [i32, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, i32, i32, dbl,
                                   _VP, i32, _VP, _VP, _VP]
            lib.orc_blocksparse.argtypes = [i32, _VP, _VP, flt, _VP, _VP, _VP, _VP, _VP, _VP]
            lib.orc_blocksparse_packed.argtypes = [i32, _VP, _VP, flt, ctypes.c_int, _VP, _VP, _VP,
                                                   _VP, _VP, _VP]
            lib.orc_order_key.restype = ctypes.c_uint32
            lib.orc_order_key.argtypes = [flt]
            lib.orc_splitmix64.restype = ctypes.c_uint64
            lib.orc_splitmix64.argtypes = [ctypes.c_uint64]
            lib.orc_perm_random.argtypes = [i32, ctypes.c_uint64, _VP]
            lib.orc_perm_degree.argtypes = [i32, _VP, _VP, _VP]
            lib.orc_perm_rcm.argtypes = [i32, _VP, _VP, _VP]
            lib.orc_apply_perm.argtypes = [i32, _VP, _VP, _VP, _VP, _VP]
            for f in ("orc_degrees", "orc_spmm", "orc_segment_reduce", "orc_gatv2",
                      "orc_gatv2_ex", "orc_gt",
                      "orc_blocksparse", "orc_perm_random", "orc_perm_degree", "orc_perm_rcm",
                      "orc_apply_perm"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _csr(rowptr, colidx):
    rp = np.ascontiguousarray(rowptr, dtype=np.int32)
    ci = np.ascontiguousarray(colidx, dtype=np.int32)
    return rp, ci, len(rp) - 1


def _feat(X):
    """(array, dtype code): fp32 -> 0, uint16 (bf16 bit patterns) -> 1."""
    if X.dtype == np.uint16:
        return np.ascontiguousarray(X), 1
    return np.ascontiguousarray(X, dtype=np.float32), 0


def _rows(rows, n):
    if rows is None:
        return None, n
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, len(r)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed ({rc})")


def degrees(rowptr, colidx, n_cols=None):
    rp, ci, n = _csr(rowptr, colidx)
    n_cols = n if n_cols is None else n_cols
    d_in = np.empty(n, np.int32)
    d_out = np.empty(n_cols, np.int32)
    _check(_load().orc_degrees(n, n_cols, _p(rp), _p(ci), _p(d_in), _p(d_out)), "degrees")
    return d_in, d_out


def spmm(rowptr, colidx, X, norm=NORM_BOTH, values=None, rows=None):
    rp, ci, n = _csr(rowptr, colidx)
    Xc, dt = _feat(X)
    F = Xc.shape[1]
    r, ns = _rows(rows, n)
    vals = None if values is None else np.ascontiguousarray(values, dtype=np.float32)
    Y = np.empty((ns, F), np.float64)
    _check(_load().orc_spmm(n, Xc.shape[0], _p(rp), _p(ci), _p(vals), norm, _p(Xc), dt, F,
                            _p(r), ns, _p(Y)), "spmm")
    return Y


def segment_reduce(op, rowptr, colidx, X, rows=None):
    """op: OP_SUM / OP_MEAN / OP_MAX / OP_MIN.  Returns Y (and the argmax or
    argmin for OP_MAX / OP_MIN)."""
    rp, ci, n = _csr(rowptr, colidx)
    Xc, dt = _feat(X)
    F = Xc.shape[1]
    r, ns = _rows(rows, n)
    Y = np.empty((ns, F), np.float64)
    am = np.empty((ns, F), np.int32) if op in (OP_MAX, OP_MIN) else None
    _check(_load().orc_segment_reduce(op, n, _p(rp), _p(ci), _p(Xc), dt, F, _p(r), ns, _p(Y),
                                      _p(am)), "segment_reduce")
    return (Y, am) if op in (OP_MAX, OP_MIN) else Y


def csr_transpose(rowptr, colidx, n_cols=None, values=None):
    """CSR^T: (rowptr_t [n_cols+1], colidx_t [nnz], values_t or None)."""
    rp, ci, n = _csr(rowptr, colidx)
    nc = n if n_cols is None else int(n_cols)
    m = len(ci)
    rpt = np.empty(nc + 1, np.int32)
    cit = np.empty(max(m, 1), np.int32)
    vals = None if values is None else np.ascontiguousarray(values, np.float32)
    vt = None if values is None else np.empty(max(m, 1), np.float32)
    _check(_load().orc_csr_transpose(n, nc, _p(rp), _p(ci), _p(vals), _p(rpt), _p(cit), _p(vt)),
           "csr_transpose")
    return rpt, cit[:m], (None if vt is None else vt[:m])


def reduce_ext_backward(arg, grad_out, n_cols):
    """Gradient of the max / min reduction w.r.t. X from the stored arg
    (argmax or argmin) and the output gradient: grad_X [n_cols, F], fp64."""
    arg = np.ascontiguousarray(arg, np.int32)
    go = np.ascontiguousarray(grad_out, np.float64)
    n_rows, F = arg.shape
    gx = np.empty((n_cols, F), np.float64)
    _check(_load().orc_reduce_ext_backward(n_rows, n_cols, F, _p(arg), _p(go), _p(gx)),
           "reduce_ext_backward")
    return gx


def gatv2(rowptr, colidx, H, W_l, a, heads, head_dim, slope=0.2, W_r=None, rows=None,
          want_alpha=False, round_c=False):
    """GATv2 forward (IO-aware GNN layers, Section 2.2 (iii), App. D.2).
    round_c: diagnostic mode, the projected features rounded to bf16 before
    the attention (as the bf16 path stores them)."""
    rp, ci, n = _csr(rowptr, colidx)
    Hc, dt = _feat(H)
    Wl, dtw = _feat(W_l)
    Wr = None if W_r is None else _feat(W_r)[0]
    if dtw != dt:
        raise ValueError("H and W must share a dtype")
    ac = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    r, ns = _rows(rows, n)
    HD = heads * head_dim
    out = np.empty((ns, HD), np.float64)
    lse = np.empty((ns, heads), np.float64)
    alpha = None
    if want_alpha:
        sel = np.arange(n) if r is None else r
        ne = int(np.sum(rp[sel + 1] - rp[sel]))
        alpha = np.empty((ne, heads), np.float64)
    _check(_load().orc_gatv2_ex(n, _p(rp), _p(ci), _p(Hc), dt, Hc.shape[1], _p(Wl), _p(Wr),
                                _p(ac), heads, head_dim, slope, _p(r), ns, int(bool(round_c)),
                                _p(out), _p(lse), _p(alpha)), "gatv2")
    return (out, lse, alpha) if want_alpha else (out, lse)


def gt(rowptr, colidx, Q, K, V, heads, head_dim, scale, rows=None, want_alpha=False):
    rp, ci, n = _csr(rowptr, colidx)
    Qc, dt = _feat(Q)
    Kc, dk = _feat(K)
    Vc, dv = _feat(V)
    if not (dt == dk == dv):
        raise ValueError("Q, K, V must share a dtype")
    r, ns = _rows(rows, n)
    HD = heads * head_dim
    out = np.empty((ns, HD), np.float64)
    lse = np.empty((ns, heads), np.float64)
    alpha = None
    if want_alpha:
        sel = np.arange(n) if r is None else r
        ne = int(np.sum(rp[sel + 1] - rp[sel]))
        alpha = np.empty((ne, heads), np.float64)
    _check(_load().orc_gt(n, _p(rp), _p(ci), _p(Qc), _p(Kc), _p(Vc), dt, heads, head_dim,
                          scale, _p(r), ns, _p(out), _p(lse), _p(alpha)), "gt")
    return (out, lse, alpha) if want_alpha else (out, lse)


def gt_backward(rowptr, colidx, Q, K, V, heads, head_dim, scale, dO):
    """Gradients (dQ, dK, dV) fp64 [n, heads*head_dim] of sum(dO * gt(...)[0])."""
    rp, ci, n = _csr(rowptr, colidx)
    Qc, dt = _feat(Q)
    Kc, _ = _feat(K)
    Vc, _ = _feat(V)
    go = np.ascontiguousarray(dO, np.float64)
    HD = heads * head_dim
    dQ, dK, dV = (np.empty((n, HD), np.float64) for _ in range(3))
    _check(_load().orc_gt_backward(n, _p(rp), _p(ci), _p(Qc), _p(Kc), _p(Vc), dt, heads, head_dim,
                                   scale, _p(go), _p(dQ), _p(dK), _p(dV)), "gt_backward")
    return dQ, dK, dV


def degree_stats(rowptr):
    """(mean, std, skewness, max) of the row lengths, population moments."""
    rp = np.ascontiguousarray(rowptr, np.int32)
    out = np.empty(4, np.float64)
    _check(_load().orc_degree_stats(len(rp) - 1, _p(rp), _p(out)), "degree_stats")
    return tuple(float(x) for x in out)


def gatv2_backward(rowptr, colidx, Cl, Cr, a, heads, head_dim, dO, slope=0.2):
    """Gradients (dl, dr fp64 [n, heads*head_dim], da fp64 [heads, head_dim])
    of sum(dO * out) for the GATv2 attention over the per-node features
    l = Cl (destination side) and r = Cr (source side); Cr=None: r = l."""
    rp, ci, n = _csr(rowptr, colidx)
    Lc, dt = _feat(Cl)
    Rc, dt_r = _feat(Cl if Cr is None else Cr)
    if dt_r != dt:
        raise TypeError("Cl and Cr must have one dtype")
    av = np.ascontiguousarray(a, np.float32)
    go = np.ascontiguousarray(dO, np.float64)
    HD = heads * head_dim
    dl, dr = (np.empty((n, HD), np.float64) for _ in range(2))
    da = np.empty((heads, head_dim), np.float64)
    _check(_load().orc_gatv2_backward(n, _p(rp), _p(ci), _p(Lc), _p(Rc), dt, _p(av), heads,
                                      head_dim, float(slope), _p(go), _p(dl), _p(dr), _p(da)),
           "gatv2_backward")
    return dl, dr, da


PACK_ID, PACK_COUNT = 0, 1


def blocksparse(rowptr, colidx, threshold, packing=PACK_ID):
    """Returns dict(grp_blk_offset, blk_cols [B,16], blk_mask [B,8,4] uint64,
    res_rowptr, res_colidx, n_tiles_kept, nnz_tiles).  packing: PACK_ID
    (columns by ascending id) or PACK_COUNT (by descending edge count in the
    group, ties by id)."""
    rp, ci, n = _csr(rowptr, colidx)
    lib = _load()
    counts = np.zeros(4, np.int64)
    _check(lib.orc_blocksparse_packed(n, _p(rp), _p(ci), float(threshold), int(packing),
                                      _p(counts), None, None, None, None, None),
           "blocksparse(count)")
    nb, nk, nt, nr = (int(x) for x in counts)
    n_groups = (n + 127) // 128
    off = np.empty(n_groups + 1, np.int32)
    cols = np.empty((nb, 16), np.int32)
    mask = np.empty((nb, 8, 4), np.uint64)
    rrp = np.empty(n + 1, np.int32)
    rci = np.empty(max(nr, 1), np.int32)
    _check(lib.orc_blocksparse_packed(n, _p(rp), _p(ci), float(threshold), int(packing),
                                      _p(counts), _p(off), _p(cols), _p(mask), _p(rrp), _p(rci)),
           "blocksparse")
    return dict(grp_blk_offset=off, blk_cols=cols, blk_mask=mask, res_rowptr=rrp,
                res_colidx=rci[:nr], n_blocks=nb, n_tiles_kept=nk, nnz_tiles=nt,
                nnz_residual=nr)


def order_key(v: float) -> int:
    return int(_load().orc_order_key(v))


def splitmix64(x: int) -> int:
    return int(_load().orc_splitmix64(x))


PERM_IDENTITY, PERM_RANDOM, PERM_DEGREE, PERM_RCM = 0, 1, 2, 3


def perm(kind, rowptr, colidx, seed=7):
    rp, ci, n = _csr(rowptr, colidx)
    out = np.empty(n, np.int32)
    lib = _load()
    if kind == PERM_IDENTITY:
        out[:] = np.arange(n, dtype=np.int32)
    elif kind == PERM_RANDOM:
        _check(lib.orc_perm_random(n, seed, _p(out)), "perm_random")
    elif kind == PERM_DEGREE:
        _check(lib.orc_perm_degree(n, _p(rp), _p(ci), _p(out)), "perm_degree")
    elif kind == PERM_RCM:
        _check(lib.orc_perm_rcm(n, _p(rp), _p(ci), _p(out)), "perm_rcm")
    else:
        raise ValueError(kind)
    return out


def apply_perm(rowptr, colidx, p):
    rp, ci, n = _csr(rowptr, colidx)
    pp = np.ascontiguousarray(p, dtype=np.int32)
    rpo = np.empty(n + 1, np.int32)
    cio = np.empty(len(ci), np.int32)
    _check(_load().orc_apply_perm(n, _p(rp), _p(ci), _p(pp), _p(rpo), _p(cio)), "apply_perm")
    return rpo, cio
