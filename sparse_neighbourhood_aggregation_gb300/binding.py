"""Thin ctypes binding of libgnn (include/gnn.h): argument marshalling only.

Every computation runs in libgnn's CUDA kernels.  PyTorch supplies device
memory (outputs, workspaces) and the current CUDA stream.  There is no CPU
fallback: if libgnn.so is missing or no GPU is visible, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("GNN_LIB_PATH") or os.path.join(_HERE, "libgnn.so")

GNN_OK, GNN_ERR_INVALID_ARG, GNN_ERR_UNSUPPORTED, GNN_ERR_WORKSPACE = 0, 1, 2, 3
GNN_ERR_CUDA, GNN_ERR_DEVICE_CHECK, GNN_ERR_TIMEOUT = 4, 5, 6
GNN_F32, GNN_BF16 = 0, 1
GNN_NORM_NONE, GNN_NORM_LEFT, GNN_NORM_RIGHT, GNN_NORM_BOTH = 0, 1, 2, 3
GNN_MAP_AUTO, GNN_MAP_FEAT, GNN_MAP_NEIGH = 0, 1, 2
(GNN_OP_SPMM, GNN_OP_SUM, GNN_OP_MEAN, GNN_OP_MAX, GNN_OP_GATV2, GNN_OP_GT, GNN_OP_REORDER,
 GNN_OP_APPLY_PERM, GNN_OP_BLOCKSPARSE, GNN_OP_MIN, GNN_OP_SPMM_BLOCKSPARSE,
 GNN_OP_TRANSPOSE, GNN_OP_GT_BACKWARD, GNN_OP_GATV2_BACKWARD, GNN_OP_GRAPH_STATS) = range(15)
GNN_BACKEND_CSR, GNN_BACKEND_TILES = 0, 1
GNN_PERM_IDENTITY, GNN_PERM_RANDOM, GNN_PERM_DEGREE, GNN_PERM_RCM = 0, 1, 2, 3
GNN_PACK_ID, GNN_PACK_COUNT = 0, 1


class GnnError(RuntimeError):
    def __init__(self, fn, code):
        msg = lib().gnn_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


class gnn_csr(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("n_cols", ctypes.c_int32), ("nnz", ctypes.c_int64),
                ("rowptr", ctypes.c_void_p), ("colidx", ctypes.c_void_p),
                ("values", ctypes.c_void_p)]


class gnn_blocksparse(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("n_blocks", ctypes.c_int64), ("n_tiles_kept", ctypes.c_int64),
                ("nnz_tiles", ctypes.c_int64), ("nnz_residual", ctypes.c_int64),
                ("fill_threshold", ctypes.c_float), ("packing", ctypes.c_int32),
                ("grp_blk_offset", ctypes.c_void_p), ("blk_cols", ctypes.c_void_p),
                ("blk_mask", ctypes.c_void_p), ("res_rowptr", ctypes.c_void_p),
                ("res_colidx", ctypes.c_void_p)]


class gnn_graph_stats(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int32), ("nnz", ctypes.c_int64), ("max_degree", ctypes.c_int32),
                ("mean_degree", ctypes.c_double), ("degree_std", ctypes.c_double),
                ("degree_skewness", ctypes.c_double), ("n_blocks", ctypes.c_int64),
                ("edges_per_block", ctypes.c_double)]


_lib = None
_lock = threading.Lock()

_SIGS = {
    "gnn_graph_prepare_size": (ctypes.c_size_t, ["csr"]),
    "gnn_graph_prepare": (ctypes.c_int, ["csr", "p", "sz", "p"]),
    "gnn_csr_validate": (ctypes.c_int, ["csr", "p"]),
    "gnn_last_device_error": (ctypes.c_int, ["p", "p"]),
    "gnn_workspace_size": (ctypes.c_size_t, ["i32", "csr", "i32", "i32", "i32"]),
    "gnn_spmm": (ctypes.c_int, ["csr", "p", "i32", "p", "i32", "i32", "p", "i32", "p", "sz", "p"]),
    "gnn_segment_reduce_sum": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p", "sz", "p"]),
    "gnn_segment_reduce_sum_noalloc": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p"]),
    "gnn_segment_reduce_mean": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p", "sz", "p"]),
    "gnn_segment_reduce_max": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p", "p", "sz",
                                              "p"]),
    "gnn_segment_reduce_min": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p", "p", "sz",
                                              "p"]),
    "gnn_segment_reduce_ext_backward": (ctypes.c_int, ["p", "i32", "i32", "p", "i32", "p", "p"]),
    "gnn_csr_transpose": (ctypes.c_int, ["csr", "p", "p", "p", "p", "sz", "p"]),
    "gnn_gt_attn_bwd": (ctypes.c_int, ["csr", "csr", "p", "p", "p", "i32", "i32", "i32", "f32", "p",
                                       "p", "p", "p", "p", "p", "p", "sz", "p"]),
    "gnn_gatv2_attn_bwd": (ctypes.c_int, ["csr", "csr", "p", "p", "i32", "p", "i32", "i32", "f32",
                                          "p", "p", "p", "p", "p", "p", "p", "sz", "p"]),
    "gnn_projection": (ctypes.c_int, ["p", "i32", "i64", "i32", "p", "i32", "p", "p"]),
    "gnn_gatv2_fwd": (ctypes.c_int, ["csr", "p", "p", "i32", "i32", "p", "p", "p", "i32", "i32",
                                     "f32", "p", "p", "p", "sz", "p"]),
    "gnn_blocksparse_plan": (ctypes.c_int, ["csr", "f32", "p", "sz", "bs", "p", "p"]),
    "gnn_blocksparse_plan_packed": (ctypes.c_int, ["csr", "f32", "i32", "p", "sz", "bs", "p", "p"]),
    "gnn_blocksparse_build": (ctypes.c_int, ["csr", "bs", "p", "sz", "p", "sz", "p"]),
    "gnn_gt_attn_fwd": (ctypes.c_int, ["csr", "p", "bs", "p", "p", "p", "i32", "i32", "i32", "f32",
                                       "p", "p", "p", "sz", "p"]),
    "gnn_spmm_blocksparse": (ctypes.c_int, ["csr", "p", "bs", "i32", "p", "i32", "i32", "p", "p",
                                            "sz", "p"]),
    "gnn_reorder_perm": (ctypes.c_int, ["csr", "i32", "u64", "p", "p", "p", "sz", "p"]),
    "gnn_apply_perm": (ctypes.c_int, ["csr", "p", "p", "p", "p", "p", "i32", "i32", "p", "p", "sz",
                                      "p"]),
    "gnn_graph_stats_compute": (ctypes.c_int, ["csr", "st", "p", "sz", "p"]),
    "gnn_select_backend": (ctypes.c_int32, ["st", "i32", "i32", "i32", "i32", "i32", "p"]),
    "gnn_status_string": (ctypes.c_char_p, ["i32"]),
    "gnn_launch_count": (ctypes.c_uint64, []),
    "gnn_version": (ctypes.c_char_p, []),
}

_CT = {"csr": ctypes.POINTER(gnn_csr), "bs": ctypes.POINTER(gnn_blocksparse),
       "st": ctypes.POINTER(gnn_graph_stats),
       "p": ctypes.c_void_p, "sz": ctypes.c_size_t, "i32": ctypes.c_int32,
       "i64": ctypes.c_int64, "u64": ctypes.c_uint64, "f32": ctypes.c_float}

EXPORTED = tuple(_SIGS)


def lib():
    """Load libgnn.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libgnn.so is not built ({LIB_PATH}); "
                                   "run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = [_CT[a] for a in args]
            _lib = L
    return _lib


def _check(name, code):
    if code != GNN_OK:
        raise GnnError(name, code)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GNN_F32
    if t.dtype == torch.bfloat16:
        return GNN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def _check_out(t: torch.Tensor, shape, dtype, device):
    """A caller-given output must match what the kernel writes."""
    if (tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device
            or not t.is_contiguous()):
        raise ValueError(f"out must be a contiguous {dtype} tensor of shape {tuple(shape)} on "
                         f"{device}; got {t.dtype} {tuple(t.shape)} on {t.device}")


class Graph:
    """A CSR graph by destination on the GPU plus its prepared buffer (step
    a0) and cached, zero-initialised workspaces."""

    def __init__(self, rowptr: torch.Tensor, colidx: torch.Tensor, values=None, n_cols=None,
                 prepare: bool = True, stream=None):
        _require_cuda(rowptr, colidx, values)
        if rowptr.dtype != torch.int32 or colidx.dtype != torch.int32:
            raise TypeError("rowptr/colidx must be int32")
        self.rowptr, self.colidx, self.values = rowptr, colidx, values
        self.n_rows = rowptr.numel() - 1
        self.n_cols = self.n_rows if n_cols is None else int(n_cols)
        self.nnz = colidx.numel()
        self.csr = gnn_csr(self.n_rows, self.n_cols, self.nnz, rowptr.data_ptr(),
                           colidx.data_ptr() if self.nnz else None, _ptr(values))
        self.device = rowptr.device
        self._ws = {}
        self.prep = None
        if prepare:
            n = lib().gnn_graph_prepare_size(ctypes.byref(self.csr))
            self.prep = torch.empty(max(n, 256), dtype=torch.uint8, device=self.device)
            _check("gnn_graph_prepare", lib().gnn_graph_prepare(
                ctypes.byref(self.csr), self.prep.data_ptr(), self.prep.numel(), _stream(stream)))

    def workspace(self, op: int, F: int = 0, heads: int = 0, head_dim: int = 0, key=None):
        n = lib().gnn_workspace_size(op, ctypes.byref(self.csr), F, heads, head_dim)
        k = (op, F, heads, head_dim, key)
        ws = self._ws.get(k)
        if ws is None or ws.numel() < n:
            ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)
            self._ws[k] = ws
        return ws


def graph_prepare(rowptr, colidx, values=None, n_cols=None, stream=None) -> Graph:
    return Graph(rowptr, colidx, values, n_cols, True, stream)


def csr_validate(g: Graph, stream=None) -> int:
    L = lib()
    _check("gnn_csr_validate", L.gnn_csr_validate(ctypes.byref(g.csr), _stream(stream)))
    code = ctypes.c_int32(0)
    _check("gnn_last_device_error", L.gnn_last_device_error(_stream(stream), ctypes.byref(code)))
    return code.value


def last_device_error(stream=None) -> int:
    """Waits for the stream, returns and clears the device error word."""
    code = ctypes.c_int32(0)
    _check("gnn_last_device_error", lib().gnn_last_device_error(_stream(stream), ctypes.byref(code)))
    return code.value


def gnn_spmm(g: Graph, X: torch.Tensor, norm: int = GNN_NORM_BOTH, mapping: int = GNN_MAP_AUTO,
             out=None, stream=None):
    _require_cuda(X)
    F = X.shape[1]
    if out is not None:
        _check_out(out, (g.n_rows, F), torch.float32, X.device)
    Y = out if out is not None else torch.empty((g.n_rows, F), dtype=torch.float32,
                                                device=X.device)
    ws = g.workspace(GNN_OP_SPMM, F)
    _check("gnn_spmm", lib().gnn_spmm(ctypes.byref(g.csr), _ptr(g.prep), norm, X.data_ptr(),
                                      _dtype_code(X), F, Y.data_ptr(), mapping, ws.data_ptr(),
                                      ws.numel(), _stream(stream)))
    return Y


def _reduce(name, op, g, X, out, stream):
    _require_cuda(X)
    F = X.shape[1]
    if out is not None:
        _check_out(out, (g.n_rows, F), torch.float32, X.device)
    Y = out if out is not None else torch.empty((g.n_rows, F), dtype=torch.float32,
                                                device=X.device)
    ws = g.workspace(op, F)
    _check(name, getattr(lib(), name)(ctypes.byref(g.csr), _ptr(g.prep), X.data_ptr(),
                                      _dtype_code(X), F, Y.data_ptr(), ws.data_ptr(), ws.numel(),
                                      _stream(stream)))
    return Y


def gnn_segment_reduce_sum(g: Graph, X, out=None, stream=None):
    return _reduce("gnn_segment_reduce_sum", GNN_OP_SUM, g, X, out, stream)


def gnn_segment_reduce_sum_noalloc(g: Graph, X, out=None, stream=None):
    """Segment sum whose scratch is the library's fixed device array instead
    of a workspace (no device allocation by the library; the output is still
    allocated here unless `out` is given)."""
    _require_cuda(X)
    F = X.shape[1]
    if out is not None:
        _check_out(out, (g.n_rows, F), torch.float32, X.device)
    # the library finds its array on the current device: make it X's
    with torch.cuda.device(X.device):
        Y = out if out is not None else torch.empty((g.n_rows, F), dtype=torch.float32,
                                                    device=X.device)
        _check("gnn_segment_reduce_sum_noalloc", lib().gnn_segment_reduce_sum_noalloc(
            ctypes.byref(g.csr), _ptr(g.prep), X.data_ptr(), _dtype_code(X), F, Y.data_ptr(),
            _stream(stream)))
    return Y


def gnn_segment_reduce_mean(g: Graph, X, out=None, stream=None):
    return _reduce("gnn_segment_reduce_mean", GNN_OP_MEAN, g, X, out, stream)


def _reduce_ext(name, op, g: Graph, X, want_arg, out, arg, stream):
    _require_cuda(X)
    F = X.shape[1]
    if out is not None:
        _check_out(out, (g.n_rows, F), torch.float32, X.device)
    if arg is not None:
        _check_out(arg, (g.n_rows, F), torch.int32, X.device)
    Y = out if out is not None else torch.empty((g.n_rows, F), dtype=torch.float32,
                                                device=X.device)
    am = None
    if want_arg:
        am = arg if arg is not None else torch.empty((g.n_rows, F), dtype=torch.int32,
                                                     device=X.device)
    ws = g.workspace(op, F)
    _check(name, getattr(lib(), name)(
        ctypes.byref(g.csr), _ptr(g.prep), X.data_ptr(), _dtype_code(X), F, Y.data_ptr(),
        _ptr(am), ws.data_ptr(), ws.numel(), _stream(stream)))
    return Y, am


def gnn_segment_reduce_max(g: Graph, X, want_argmax: bool = True, out=None, argmax=None,
                           stream=None):
    return _reduce_ext("gnn_segment_reduce_max", GNN_OP_MAX, g, X, want_argmax, out, argmax,
                       stream)


def gnn_segment_reduce_min(g: Graph, X, want_argmin: bool = True, out=None, argmin=None,
                           stream=None):
    return _reduce_ext("gnn_segment_reduce_min", GNN_OP_MIN, g, X, want_argmin, out, argmin,
                       stream)


def launch_count() -> int:
    return int(lib().gnn_launch_count())


def version() -> str:
    return lib().gnn_version().decode()


GNN_OP_FLAG_BF16 = 0x100


def _ws_op(op: int, t: torch.Tensor) -> int:
    return op | (GNN_OP_FLAG_BF16 if t.dtype == torch.bfloat16 else 0)


def gnn_projection(H: torch.Tensor, W: torch.Tensor, out=None, stream=None):
    """C = H W (bf16: tcgen05 tensor cores, fp32 accumulation, bf16 out;
    fp32: fp32 FMA)."""
    _require_cuda(H, W)
    n, F_in = H.shape
    F_out = W.shape[1]
    C = out if out is not None else torch.empty((n, F_out), dtype=H.dtype, device=H.device)
    _check("gnn_projection", lib().gnn_projection(H.data_ptr(), _dtype_code(H), n, F_in,
                                                  W.data_ptr(), F_out, C.data_ptr(),
                                                  _stream(stream)))
    return C


def gnn_gatv2_fwd(g: Graph, H: torch.Tensor, W_l: torch.Tensor, a: torch.Tensor, heads: int,
                  head_dim: int, neg_slope: float = 0.2, W_r=None, want_lse: bool = True,
                  out=None, lse=None, stream=None):
    """Fused GATv2 forward: returns (out [n, heads*head_dim] fp32, lse [n,
    heads] fp32 or None)."""
    _require_cuda(H, W_l, W_r, a)
    if a.dtype != torch.float32:
        raise TypeError("a must be fp32")
    HD = heads * head_dim
    o = out if out is not None else torch.empty((g.n_rows, HD), dtype=torch.float32,
                                                device=H.device)
    L = None
    if want_lse:
        L = lse if lse is not None else torch.empty((g.n_rows, heads), dtype=torch.float32,
                                                    device=H.device)
    ws = g.workspace(_ws_op(GNN_OP_GATV2, H), H.shape[1], heads, head_dim)
    _check("gnn_gatv2_fwd", lib().gnn_gatv2_fwd(
        ctypes.byref(g.csr), _ptr(g.prep), H.data_ptr(), _dtype_code(H), H.shape[1],
        W_l.data_ptr(), _ptr(W_r), a.data_ptr(), heads, head_dim, float(neg_slope),
        o.data_ptr(), _ptr(L), ws.data_ptr(), ws.numel(), _stream(stream)))
    return o, L


def gnn_gt_attn_fwd(g: Graph, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, heads: int,
                    head_dim: int, scale: float, bs=None, want_lse: bool = True, out=None,
                    lse=None, stream=None):
    """Graph Transformer attention: returns (out fp32 [n, heads*head_dim],
    lse fp32 [n, heads] or None).  bs: a BlockSparse from
    gnn_blocksparse_build for the tensor-core tile path, or None (CSR)."""
    _require_cuda(Q, K, V)
    HD = heads * head_dim
    o = out if out is not None else torch.empty((g.n_rows, HD), dtype=torch.float32,
                                                device=Q.device)
    L = None
    if want_lse:
        L = lse if lse is not None else torch.empty((g.n_rows, heads), dtype=torch.float32,
                                                    device=Q.device)
    ws = g.workspace(_ws_op(GNN_OP_GT, Q), 0, heads, head_dim, key="bs" if bs is not None else None)
    bsp = ctypes.byref(bs.meta) if bs is not None else None
    _check("gnn_gt_attn_fwd", lib().gnn_gt_attn_fwd(
        ctypes.byref(g.csr), _ptr(g.prep), bsp, Q.data_ptr(), K.data_ptr(), V.data_ptr(),
        _dtype_code(Q), heads, head_dim, float(scale), o.data_ptr(), _ptr(L), ws.data_ptr(),
        ws.numel(), _stream(stream)))
    return o, L


def gnn_segment_reduce_ext_backward(arg: torch.Tensor, grad_out: torch.Tensor, n_cols: int,
                                    out=None, stream=None):
    """Gradient w.r.t. X of gnn_segment_reduce_max / _min from their arg
    output and the output gradient: grad_X fp32 [n_cols, F]."""
    _require_cuda(arg, grad_out)
    n_rows, F = arg.shape
    gx = out if out is not None else torch.empty((n_cols, F), dtype=torch.float32,
                                                 device=arg.device)
    _check("gnn_segment_reduce_ext_backward", lib().gnn_segment_reduce_ext_backward(
        arg.data_ptr(), n_rows, F, grad_out.data_ptr(), n_cols, gx.data_ptr(), _stream(stream)))
    return gx


def gnn_csr_transpose(g: Graph, stream=None):
    """CSR^T of g: returns (rowptr_t [n_cols+1], colidx_t [nnz], values_t or
    None) int32 / fp32 tensors; prepare the result with graph_prepare to run
    the backward of gnn_spmm as a gnn_spmm on it."""
    rp = torch.empty(g.csr.n_cols + 1, dtype=torch.int32, device=g.device)
    ci = torch.empty(max(g.csr.nnz, 1), dtype=torch.int32, device=g.device)[:g.csr.nnz]
    vals = None
    if g.csr.values:
        vals = torch.empty(max(g.csr.nnz, 1), dtype=torch.float32, device=g.device)[:g.csr.nnz]
    ws = g.workspace(GNN_OP_TRANSPOSE)
    _check("gnn_csr_transpose", lib().gnn_csr_transpose(
        ctypes.byref(g.csr), rp.data_ptr(), ci.data_ptr() if g.csr.nnz else None, _ptr(vals),
        ws.data_ptr(), ws.numel(), _stream(stream)))
    return rp, ci, vals


def gnn_gt_attn_bwd(g: Graph, gt: Graph, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                    heads: int, head_dim: int, scale: float, out: torch.Tensor, lse: torch.Tensor,
                    dout: torch.Tensor, stream=None):
    """Backward of gnn_gt_attn_fwd (CSR path): returns (dQ, dK, dV) fp32.
    gt: the transpose of g (Graph over gnn_csr_transpose's arrays)."""
    _require_cuda(Q, K, V, out, lse, dout)
    HD = heads * head_dim
    dQ, dK, dV = (torch.empty((g.n_rows, HD), dtype=torch.float32, device=Q.device)
                  for _ in range(3))
    ws = g.workspace(GNN_OP_GT_BACKWARD, 0, heads, head_dim)
    _check("gnn_gt_attn_bwd", lib().gnn_gt_attn_bwd(
        ctypes.byref(g.csr), ctypes.byref(gt.csr), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
        _dtype_code(Q), heads, head_dim, float(scale), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(stream)))
    return dQ, dK, dV


def gnn_gatv2_attn_bwd(g: Graph, gt: Graph, Cl: torch.Tensor, Cr, a: torch.Tensor, heads: int,
                       head_dim: int, out: torch.Tensor, lse: torch.Tensor, dout: torch.Tensor,
                       neg_slope: float = 0.2, stream=None):
    """Backward of the GATv2 attention over the projected features: returns
    (dl, dr fp32 [n, heads*head_dim], da fp32 [heads, head_dim]).  Cl: the
    destination-side features l; Cr: the source-side features r (None: one
    projection, r = l, whose gradient is dl + dr).  gt: the transpose of g."""
    Cr = Cl if Cr is None else Cr
    _require_cuda(Cl, Cr, a, out, lse, dout)
    if a.dtype != torch.float32 or Cr.dtype != Cl.dtype:
        raise TypeError("a must be fp32 and Cl, Cr of one dtype")
    HD = heads * head_dim
    dl, dr = (torch.empty((g.n_rows, HD), dtype=torch.float32, device=Cl.device) for _ in range(2))
    da = torch.empty((heads, head_dim), dtype=torch.float32, device=Cl.device)
    ws = g.workspace(GNN_OP_GATV2_BACKWARD, 0, heads, head_dim)
    _check("gnn_gatv2_attn_bwd", lib().gnn_gatv2_attn_bwd(
        ctypes.byref(g.csr), ctypes.byref(gt.csr), Cl.data_ptr(), Cr.data_ptr(), _dtype_code(Cl),
        a.data_ptr(), heads, head_dim, float(neg_slope), out.data_ptr(), lse.data_ptr(),
        dout.data_ptr(), dl.data_ptr(), dr.data_ptr(), da.data_ptr(), ws.data_ptr(), ws.numel(),
        _stream(stream)))
    return dl, dr, da


def gnn_graph_stats_compute(g: Graph, stream=None) -> gnn_graph_stats:
    """Degree moments and local density of g, measured on the GPU
    (synchronous); returns the filled gnn_graph_stats."""
    st = gnn_graph_stats()
    ws = g.workspace(GNN_OP_GRAPH_STATS)
    _check("gnn_graph_stats_compute", lib().gnn_graph_stats_compute(
        ctypes.byref(g.csr), ctypes.byref(st), ws.data_ptr(), ws.numel(), _stream(stream)))
    return st


def gnn_select_backend(stats: gnn_graph_stats, op: int, dtype: int, F: int = 0, heads: int = 0,
                       head_dim: int = 0):
    """Host rule: (GNN_BACKEND_CSR or GNN_BACKEND_TILES, fill threshold for
    the tile build) for op GNN_OP_SPMM or GNN_OP_GT.  No GPU work."""
    thr = ctypes.c_float(0.0)
    b = lib().gnn_select_backend(ctypes.byref(stats), int(op), int(dtype), int(F), int(heads),
                                 int(head_dim), ctypes.byref(thr))
    return int(b), float(thr.value)


def gnn_spmm_blocksparse(g: Graph, X: torch.Tensor, bs, norm: int = GNN_NORM_BOTH, out=None,
                         stream=None):
    """GCN SpMM over a BlockSparse from gnn_blocksparse_build: kept tiles on
    the tensor cores, residual edges on the CSR kernel.  X bf16 [n_cols, F],
    F a multiple of 64; returns Y fp32 [n_rows, F]."""
    _require_cuda(X)
    F = X.shape[1]
    Y = out if out is not None else torch.empty((g.n_rows, F), dtype=torch.float32, device=X.device)
    ws = g.workspace(GNN_OP_SPMM_BLOCKSPARSE, F, key=("bs", int(bs.meta.nnz_residual)))
    _check("gnn_spmm_blocksparse", lib().gnn_spmm_blocksparse(
        ctypes.byref(g.csr), _ptr(g.prep), ctypes.byref(bs.meta), int(norm), X.data_ptr(),
        _dtype_code(X), F, Y.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream)))
    return Y


def gnn_reorder_perm(g: Graph, kind: int, seed: int = 7, stream=None):
    """Vertex order of a square graph: returns (perm, inv) int32 tensors,
    perm[new] = old, inv[old] = new.  RCM is synchronous."""
    perm = torch.empty(g.n_rows, dtype=torch.int32, device=g.device)
    inv = torch.empty(g.n_rows, dtype=torch.int32, device=g.device)
    ws = g.workspace(GNN_OP_REORDER)
    _check("gnn_reorder_perm", lib().gnn_reorder_perm(ctypes.byref(g.csr), int(kind), int(seed),
                                                      perm.data_ptr(), inv.data_ptr(),
                                                      ws.data_ptr(), ws.numel(), _stream(stream)))
    return perm, inv


def gnn_apply_perm(g: Graph, perm: torch.Tensor, inv=None, X=None, stream=None):
    """Relabel g by perm (perm[new] = old): returns (rowptr, colidx, X_out)
    with columns re-sorted within rows and X_out[r] = X[perm[r]] (None if X
    is None)."""
    _require_cuda(perm, inv, X)
    rp = torch.empty(g.n_rows + 1, dtype=torch.int32, device=g.device)
    ci = torch.empty(max(g.nnz, 1), dtype=torch.int32, device=g.device)
    Xo = None
    if X is not None:
        Xo = torch.empty_like(X)
    ws = g.workspace(GNN_OP_APPLY_PERM)
    _check("gnn_apply_perm", lib().gnn_apply_perm(
        ctypes.byref(g.csr), perm.data_ptr(), _ptr(inv), rp.data_ptr(), ci.data_ptr(), _ptr(X),
        _dtype_code(X) if X is not None else 0, X.shape[1] if X is not None else 0, _ptr(Xo),
        ws.data_ptr(), ws.numel(), _stream(stream)))
    return rp, ci[:g.nnz], Xo


class BlockSparse:
    """A built block-sparse layout (step a6): the host descriptor `meta`
    (gnn_blocksparse) and the device buffer that holds its arrays."""

    def __init__(self, meta: gnn_blocksparse, buf: torch.Tensor):
        self.meta, self.buf = meta, buf

    def _view(self, ptr, count, dtype):
        if count == 0:
            return torch.empty(0, dtype=dtype, device=self.buf.device)
        off = ptr - self.buf.data_ptr()
        nbytes = count * torch.empty(0, dtype=dtype).element_size()
        return self.buf[off:off + nbytes].view(dtype)

    def arrays(self):
        m = self.meta
        return {"grp_blk_offset": self._view(m.grp_blk_offset, m.n_groups + 1, torch.int32),
                "blk_cols": self._view(m.blk_cols, m.n_blocks * 16, torch.int32).view(-1, 16),
                "blk_mask": self._view(m.blk_mask, m.n_blocks * 32, torch.int64).view(-1, 8, 4),
                "res_rowptr": self._view(m.res_rowptr, m.n_rows + 1, torch.int32),
                "res_colidx": self._view(m.res_colidx, m.nnz_residual, torch.int32)}


def gnn_blocksparse_build(g: Graph, fill_threshold: float, packing: int = 0,
                          stream=None) -> BlockSparse:
    """Plan and build the 16x16 block-sparse tile layout of g (synchronous).
    packing: GNN_PACK_ID (columns by id) or GNN_PACK_COUNT (by descending
    edge count in the group)."""
    ws = g.workspace(GNN_OP_BLOCKSPARSE)
    meta = gnn_blocksparse()
    nbytes = ctypes.c_size_t(0)
    L = lib()
    _check("gnn_blocksparse_plan_packed", L.gnn_blocksparse_plan_packed(
        ctypes.byref(g.csr), float(fill_threshold), int(packing), ws.data_ptr(), ws.numel(),
        ctypes.byref(meta), ctypes.byref(nbytes), _stream(stream)))
    buf = torch.empty(max(nbytes.value, 256), dtype=torch.uint8, device=g.device)
    _check("gnn_blocksparse_build", L.gnn_blocksparse_build(
        ctypes.byref(g.csr), ctypes.byref(meta), buf.data_ptr(), buf.numel(), ws.data_ptr(),
        ws.numel(), _stream(stream)))
    return BlockSparse(meta, buf)
