"""GPU parity of the graph statistics the backend choice reads (degree
moments and the block-sparse plan's block count) against the CPU oracle,
through the C ABI, and the choice on the clustered and power-law graphs.
Marked gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G

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


def check_stats(gnn, rp, ci):
    g = gnn.Graph(dev(rp), dev(ci), None, None, False)
    st = gnn.gnn_graph_stats_compute(g)
    mean, std, skew, mx = oracle.degree_stats(rp)
    nb = oracle.blocksparse(rp, ci, 0.0)["n_blocks"]
    assert (st.n_rows, st.nnz, st.max_degree, st.n_blocks) == (len(rp) - 1, len(ci), int(mx), nb)
    # exact integer moments on the GPU against the oracle's sequential fp64
    # two-pass sums: a sum of n terms carries at most n ulps of the sum of
    # their magnitudes (Higham, the recursive-summation bound), so the
    # tolerances scale with n and, for the third moment, with sum |c|^3
    n = len(rp) - 1
    eps = 8 * n * 2.0 ** -53
    c = np.diff(rp).astype(np.float64) - mean
    m2 = std * std
    assert st.mean_degree == pytest.approx(mean, rel=1e-15)
    assert st.degree_std == pytest.approx(std, rel=eps, abs=1e-12)
    tol_skew = eps * np.mean(np.abs(c) ** 3) / m2 ** 1.5 + eps * abs(skew) if m2 > 0 else 1e-12
    assert st.degree_skewness == pytest.approx(skew, rel=0, abs=tol_skew)
    assert st.edges_per_block == pytest.approx(len(ci) / nb if nb else 0.0, rel=1e-15)
    return st


def test_stats_small_graphs(gnn):
    for rp, ci in [G.star(300), G.grid(20), G.path(50), G.random_graph(60, 0.1, 2),
                   G.from_edges(40, [(1, 2), (3, 2), (5, 9)], self_loops=False)]:
        check_stats(gnn, rp, ci)


def test_stats_regular_graph_has_no_spread(gnn):
    rp, ci = G.from_edges(64, [((i + k) % 64, i) for i in range(64) for k in range(1, 6)],
                          self_loops=False)
    st = check_stats(gnn, rp, ci)
    assert (st.degree_std, st.degree_skewness) == (0.0, 0.0)


def test_stats_and_choice_on_the_workload_graphs(gnn):
    """R-MAT scale 17 (power law, a few edges per block) runs on CSR; the
    clustered 262K-node graph (about 440 edges per block) on the tiles."""
    w = synth.workload("c2_rmat17", features=False)
    st = check_stats(gnn, w["rowptr"], w["colidx"])
    assert st.degree_skewness > 10
    assert gnn.gnn_select_backend(st, gnn.GNN_OP_SPMM, gnn.GNN_BF16, 256)[0] == gnn.GNN_BACKEND_CSR
    w = synth.workload("c4_clustered_gt", features=False)
    st = check_stats(gnn, w["rowptr"], w["colidx"])
    assert gnn.gnn_select_backend(st, gnn.GNN_OP_SPMM, gnn.GNN_BF16, 256) == (gnn.GNN_BACKEND_TILES, 0.0)
    assert gnn.gnn_select_backend(st, gnn.GNN_OP_GT, gnn.GNN_BF16, 0, 8, 32)[0] == gnn.GNN_BACKEND_TILES
