"""GPU parity of the CSR^T build and of the SpMM backward run as a SpMM on
CSR^T, against the CPU oracle, through the C ABI.  Marked gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G
from tests.tolerance import TOL_F32, assert_rowwise_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gnn():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test was selected but torch sees no CUDA device")
    import sparse_neighbourhood_aggregation_gb300 as m
    m.lib()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_transpose(gnn, rp, ci, n_cols=None, values=None):
    g = gnn.Graph(dev(rp), dev(ci), None if values is None else dev(values), n_cols, False)
    rpt, cit, vt = gnn.gnn_csr_transpose(g)
    erp, eci, ev = oracle.csr_transpose(rp, ci, n_cols=n_cols, values=values)
    assert np.array_equal(rpt.cpu().numpy(), erp), "rowptr_t"
    assert np.array_equal(cit.cpu().numpy(), eci), "colidx_t"
    if values is not None:
        assert np.array_equal(vt.cpu().numpy(), ev), "values_t"
    return rpt, cit


def test_transpose_small_graphs(gnn):
    for rp, ci in [G.random_graph(7, 0.3, 0), G.star(17), G.path(40), G.grid(9),
                   G.from_edges(9, [], self_loops=False)]:
        check_transpose(gnn, rp, ci)


def test_transpose_rectangular_with_values(gnn):
    rng = np.random.default_rng(3)
    n_rows, n_cols = 300, 1000
    deg = rng.integers(0, 20, n_rows)
    rp = np.zeros(n_rows + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    ci = np.concatenate([np.sort(rng.choice(n_cols, d, replace=False)) for d in deg]).astype(np.int32)
    vals = rng.standard_normal(len(ci)).astype(np.float32)
    check_transpose(gnn, rp, ci, n_cols=n_cols, values=vals)


def test_transpose_config2(gnn):
    w = synth.workload("c2_rmat17", features=False)
    check_transpose(gnn, w["rowptr"], w["colidx"])


@pytest.mark.parametrize("norm,bnorm", [(3, 3), (1, 2)])
def test_spmm_backward_on_the_transpose_config2(gnn, norm, bnorm):
    """GCN (BOTH) and mean (LEFT) SpMM backward on R-MAT scale 17: the GPU
    SpMM on the GPU-built CSR^T (norm BOTH / RIGHT) against the oracle's
    SpMM on its own CSR^T."""
    w = synth.workload("c2_rmat17", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n = len(rp) - 1
    g = gnn.Graph(dev(rp), dev(ci), None, None, False)
    rpt, cit, _ = gnn.gnn_csr_transpose(g)
    gt = gnn.graph_prepare(rpt, cit)
    gy = synth.normal_f32((n, 128), 1.0, 61)
    got = gnn.gnn_spmm(gt, dev(gy), norm=bnorm).cpu().numpy()
    erp, eci, _ = oracle.csr_transpose(rp, ci)
    rows = np.unique(np.concatenate([np.random.default_rng(2).choice(n, 400, replace=False),
                                     np.argsort(-np.diff(erp))[:8]])).astype(np.int32)
    ref = oracle.spmm(erp, eci, gy, norm=bnorm, rows=rows)
    assert_rowwise_close(got[rows], ref, TOL_F32, f"spmm backward norm={norm}")
