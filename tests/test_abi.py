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
