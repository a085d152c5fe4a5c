"""GPU parity of the CSR^T build and of the SpMM backward run as a SpMM on
CSR^T, against the CPU oracle, through the C ABI.  Marked gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G
from tests.tolerance import TOL_BF16, TOL_F32, assert_rowwise_close

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


def _bf16(shape, seed):
    return synth.normal_bf16(shape, 1.0, seed)


def check_gt_backward(gnn, rp, ci, heads, D, seed=0):
    n = len(rp) - 1
    HD = heads * D
    Q, K, V = (_bf16((n, HD), 70 + 3 * seed + k) for k in range(3))
    dO = synth.normal_f32((n, HD), 1.0, 80 + seed)
    scale = 1.0 / np.sqrt(D)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    qd, kd, vd = (dev(x.view(np.int16)).view(torch.bfloat16) for x in (Q, K, V))
    out, lse = gnn.gnn_gt_attn_fwd(g, qd, kd, vd, heads, D, scale)
    rpt, cit, _ = gnn.gnn_csr_transpose(gnn.Graph(dev(rp), dev(ci), None, None, False))
    gt = gnn.Graph(rpt, cit, None, None, False)
    dQ, dK, dV = gnn.gnn_gt_attn_bwd(g, gt, qd, kd, vd, heads, D, scale, out, lse, dev(dO))
    rQ, rK, rV = oracle.gt_backward(rp, ci, Q, K, V, heads, D, scale, dO)
    for got, ref, name in ((dQ, rQ, "dQ"), (dK, rK, "dK"), (dV, rV, "dV")):
        assert_rowwise_close(got.cpu().numpy(), ref, TOL_BF16, f"gt backward {name} {heads}x{D}")


@pytest.mark.parametrize("heads,D", [(8, 32), (4, 64), (4, 32), (2, 64)])
def test_gt_backward_small_graphs(gnn, heads, D):
    rng = np.random.default_rng(heads * D)
    n = 400
    edges = [(int(rng.integers(n)), int(rng.integers(n))) for _ in range(6 * n)]
    edges += [(int(s), 7) for s in rng.choice(n, 300, replace=False)]  # a hub destination
    edges += [(3, int(d)) for d in rng.choice(n, 200, replace=False)]  # a hub source
    rp, ci = G.from_edges(n, [(s, d) for s, d in edges if d not in (50, 51)], self_loops=False)
    check_gt_backward(gnn, rp, ci, heads, D)


def test_gt_backward_clustered(gnn):
    rp, ci = synth.clustered(32, 128, 0.3, 0.02, 5)
    check_gt_backward(gnn, rp, ci, 8, 32, seed=1)


def test_gt_backward_rejects_unsupported_shapes(gnn):
    rp, ci = G.random_graph(20, 0.2, 1)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    gt = gnn.Graph(*gnn.gnn_csr_transpose(g)[:2], None, None, False)
    x = torch.zeros((20, 96), dtype=torch.bfloat16, device="cuda")
    f = torch.zeros((20, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_gt_attn_bwd(g, gt, x, x, x, 3, 32, 0.2, f, torch.zeros((20, 3), device="cuda"), f)
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED
