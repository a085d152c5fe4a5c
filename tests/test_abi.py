"""The C-ABI library loads, exports every entry point include/gnn.h
declares, and rejects bad arguments on the host before touching the GPU.
CPU only: no call here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gnn.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gnn_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from sparse_neighbourhood_aggregation_gb300 import _build, binding
    _build.build()
    return binding.lib()


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for required in ["gnn_spmm", "gnn_segment_reduce_sum", "gnn_segment_reduce_mean",
                     "gnn_segment_reduce_max", "gnn_gatv2_fwd", "gnn_gt_attn_fwd",
                     "gnn_reorder_perm", "gnn_blocksparse_build", "gnn_graph_prepare",
                     "gnn_projection", "gnn_apply_perm"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from sparse_neighbourhood_aggregation_gb300 import binding
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.EXPORTED, f"binding lacks a signature for {name}"


def test_host_side_calls(lib):
    from sparse_neighbourhood_aggregation_gb300 import binding as b
    assert lib.gnn_status_string(b.GNN_ERR_WORKSPACE) == b"workspace too small"
    assert b"sm_103a" in lib.gnn_version()
    # invalid arguments are rejected before any CUDA call
    assert lib.gnn_spmm(None, None, 0, None, 0, 32, None, 0, None, 0, None) == b.GNN_ERR_INVALID_ARG
    csr = b.gnn_csr(4, 4, 2**31, 1, 1, None)      # nnz beyond int32
    assert lib.gnn_segment_reduce_sum(ctypes.byref(csr), None, 1, 0, 32, 1, None, 0, None) == \
        b.GNN_ERR_INVALID_ARG
    csr = b.gnn_csr(1000, 1000, 5000, 16, 16, None)
    assert lib.gnn_graph_prepare_size(ctypes.byref(csr)) >= 1000 * 4 * 3
    assert lib.gnn_workspace_size(b.GNN_OP_MAX, ctypes.byref(csr), 128, 0, 0) > \
        lib.gnn_workspace_size(b.GNN_OP_SUM, ctypes.byref(csr), 128, 0, 0)
    # unsupported widths: F=12 fp32 is three 16-byte chunks
    assert lib.gnn_spmm(ctypes.byref(csr), None, 0, 16, 0, 12, 16, 0, None, 0, None) == \
        b.GNN_ERR_UNSUPPORTED


def test_select_backend_rule(lib):
    """The backend rule is host code: no GPU.  Local density at or above the
    measured break-even (158 edges a block for SpMM, 129 for GT) picks the
    tiles when the inputs qualify; everything else runs on CSR."""
    import oracle
    import synth
    from sparse_neighbourhood_aggregation_gb300 import binding as b

    def stats(epb, nnz=1000):
        return b.gnn_graph_stats(n_rows=100, nnz=nnz, max_degree=10, mean_degree=10.0,
                                 degree_std=1.0, degree_skewness=0.0, n_blocks=max(1, int(nnz / epb)),
                                 edges_per_block=epb)

    sp, gt = b.GNN_OP_SPMM, b.GNN_OP_GT
    assert b.gnn_select_backend(stats(439.0), sp, b.GNN_BF16, 256) == (b.GNN_BACKEND_TILES, 0.0)
    assert b.gnn_select_backend(stats(158.0), sp, b.GNN_BF16, 64)[0] == b.GNN_BACKEND_TILES
    assert b.gnn_select_backend(stats(157.9), sp, b.GNN_BF16, 64)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(439.0), sp, b.GNN_F32, 256)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(439.0), sp, b.GNN_BF16, 96)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(130.0), gt, b.GNN_BF16, 0, 8, 32)[0] == b.GNN_BACKEND_TILES
    assert b.gnn_select_backend(stats(128.0), gt, b.GNN_BF16, 0, 8, 32)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(439.0), gt, b.GNN_BF16, 0, 2, 128)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(439.0), b.GNN_OP_MAX, b.GNN_BF16, 256)[0] == b.GNN_BACKEND_CSR
    assert b.gnn_select_backend(stats(439.0, nnz=0), sp, b.GNN_BF16, 256)[0] == b.GNN_BACKEND_CSR
    # on densities the oracle measures: a clustered graph qualifies, R-MAT does not
    for (rp, ci), want in ((synth.clustered(8, 128, 0.3, 0.01, 3), b.GNN_BACKEND_TILES),
                           (synth.rmat(12, 16), b.GNN_BACKEND_CSR)):
        nb = oracle.blocksparse(rp, ci, 0.0)["n_blocks"]
        s = stats(len(ci) / nb, nnz=len(ci))
        assert b.gnn_select_backend(s, sp, b.GNN_BF16, 256)[0] == want
        assert b.gnn_select_backend(s, gt, b.GNN_BF16, 0, 8, 32)[0] == want


def test_backward_and_statistics_host_validation(lib):
    """The GATv2 backward and the statistics call reject bad arguments and
    short workspaces on the host, before any CUDA call."""
    from sparse_neighbourhood_aggregation_gb300 import binding as b
    sq = b.gnn_csr(1000, 1000, 5000, 16, 16, None)
    rect = b.gnn_csr(1000, 900, 5000, 16, 16, None)
    other = b.gnn_csr(1000, 1000, 4000, 16, 16, None)
    P = 4096  # a 16-byte aligned stand-in for a device pointer (never dereferenced)

    def bwd(g, gt, dtype=b.GNN_BF16, heads=4, D=64, a=P, dl=P, ws=P, ws_bytes=1 << 40):
        return lib.gnn_gatv2_attn_bwd(None if g is None else ctypes.byref(g), ctypes.byref(gt), P, P,
                                      dtype, a, heads, D, 0.2, P, P, P, dl, P, P, ws, ws_bytes, None)

    assert bwd(None, sq) == b.GNN_ERR_INVALID_ARG
    assert bwd(rect, sq) == b.GNN_ERR_INVALID_ARG          # not square
    assert bwd(sq, other) == b.GNN_ERR_INVALID_ARG         # transpose of another graph
    assert bwd(sq, sq, dtype=7) == b.GNN_ERR_UNSUPPORTED
    assert bwd(sq, sq, heads=3, D=32) == b.GNN_ERR_UNSUPPORTED   # 96 channels
    assert bwd(sq, sq, heads=64, D=4) == b.GNN_ERR_UNSUPPORTED   # 8 channels a lane, heads of 4
    assert bwd(sq, sq, a=None) == b.GNN_ERR_INVALID_ARG
    assert bwd(sq, sq, dl=P + 4) == b.GNN_ERR_INVALID_ARG        # dl not 16-byte aligned
    assert bwd(sq, sq, ws_bytes=0) == b.GNN_ERR_WORKSPACE
    need = lib.gnn_workspace_size(b.GNN_OP_GATV2_BACKWARD, ctypes.byref(sq), 0, 4, 64)
    assert need > lib.gnn_workspace_size(b.GNN_OP_GATV2_BACKWARD, ctypes.byref(sq), 0, 1, 32) > 0
    assert bwd(sq, sq, ws_bytes=need - 1) == b.GNN_ERR_WORKSPACE

    st = b.gnn_graph_stats()
    assert lib.gnn_graph_stats_compute(None, ctypes.byref(st), P, 1 << 40, None) == b.GNN_ERR_INVALID_ARG
    assert lib.gnn_graph_stats_compute(ctypes.byref(sq), None, P, 1 << 40, None) == b.GNN_ERR_INVALID_ARG
    assert lib.gnn_graph_stats_compute(ctypes.byref(sq), ctypes.byref(st), P, 0, None) == \
        b.GNN_ERR_WORKSPACE
    assert lib.gnn_workspace_size(b.GNN_OP_GRAPH_STATS, ctypes.byref(sq), 0, 0, 0) > 0
    empty = b.gnn_csr(0, 0, 0, 16, None, None)
    assert lib.gnn_graph_stats_compute(ctypes.byref(empty), ctypes.byref(st), None, 0, None) == b.GNN_OK
    assert (st.n_rows, st.nnz, st.n_blocks, st.edges_per_block) == (0, 0, 0, 0.0)
    assert lib.gnn_select_backend(None, b.GNN_OP_SPMM, b.GNN_BF16, 256, 0, 0, None) == b.GNN_BACKEND_CSR
