"""GPU parity of the tensor-core SpMM over block-sparse tiles (kept tiles on
tcgen05, residual edges on the CSR kernel) against the CPU oracle's SpMM,
through the C ABI.  Marked gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G
from tests.tolerance import TOL_BF16, assert_rowwise_close

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
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def check(gnn, rp, ci, X, thr, norms=(0, 1, 2, 3), rows=None, packing=0):
    g = gnn.graph_prepare(dev(rp), dev(ci))
    bs = gnn.gnn_blocksparse_build(g, thr, packing=packing)
    Xd = dev(X)
    sel = slice(None) if rows is None else rows
    for norm in norms:
        Y = gnn.gnn_spmm_blocksparse(g, Xd, bs, norm=norm).cpu().numpy()
        ref = oracle.spmm(rp, ci, X, norm=norm, rows=rows)
        assert_rowwise_close(Y[sel], ref, TOL_BF16, f"tile spmm thr={thr} norm={norm}")
    return bs


@pytest.mark.parametrize("thr", [0.0, 0.3, 1.0])
@pytest.mark.parametrize("F", [64, 256])
def test_clustered_all_norms(gnn, thr, F):
    # 6 clusters of 96 nodes: dense diagonal tiles, rewired edges in sparse
    # tiles or the residual, a ragged last row group
    rp, ci = synth.clustered(6, 96, 0.3, 0.05, 3)
    n = len(rp) - 1
    X = synth.normal_bf16((n, F), 1.0, 40)
    bs = check(gnn, rp, ci, X, thr)
    if thr == 0.0:
        assert bs.meta.nnz_residual == 0
    if thr == 1.0:
        assert bs.meta.nnz_residual > 0


def test_empty_groups_and_rows(gnn):
    """Row groups 1 and 3 have no edges and single rows inside tiled groups
    have none either: zero rows, with and without residual edges."""
    n = 600
    rng = np.random.default_rng(21)
    empty = set(range(128, 256)) | set(range(384, 512)) | {5, 70, 300, 599}
    edges = [(int(rng.integers(n)), d) for d in range(n) if d not in empty for _ in range(6)]
    rp, ci = G.from_edges(n, edges, self_loops=False)
    X = synth.normal_bf16((n, 128), 1.0, 41)
    for thr in (0.0, 0.5):
        check(gnn, rp, ci, X, thr)


def test_dense_clique_full_tiles(gnn):
    # a 64-node clique fills whole tiles; a ring adds residual edges
    rp, ci = G.from_edges(200, [(a, b) for a in range(64) for b in range(64)] +
                          [(i, (i + 1) % 200) for i in range(200)])
    X = synth.normal_bf16((200, 64), 1.0, 42)
    for thr in (0.0, 0.9):
        check(gnn, rp, ci, X, thr)


def test_config4_graph_sampled(gnn):
    w = synth.workload("c4_clustered_gt", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n = len(rp) - 1
    X = synth.normal_bf16((n, 256), 1.0, 43)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rng.choice(n, 200, replace=False),
                                     [0, 127, 128, n - 1]])).astype(np.int32)
    for thr in (0.0, 0.2):
        check(gnn, rp, ci, X, thr, norms=(0, 3), rows=rows)
    # columns in count-sorted order
    for thr in (0.0, 0.3):
        check(gnn, rp, ci, X, thr, norms=(3,), rows=rows, packing=1)


@pytest.mark.parametrize("thr", [0.0, 0.3, 0.4])
def test_count_packing_clustered(gnn, thr):
    rp, ci = synth.clustered(6, 96, 0.3, 0.05, 4)
    n = len(rp) - 1
    X = synth.normal_bf16((n, 128), 1.0, 45)
    check(gnn, rp, ci, X, thr, packing=1)


def test_rejects_unsupported_inputs(gnn):
    rp, ci = synth.clustered(2, 64, 0.3, 0.0, 1)
    n = len(rp) - 1
    g = gnn.graph_prepare(dev(rp), dev(ci))
    bs = gnn.gnn_blocksparse_build(g, 0.0)
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_spmm_blocksparse(g, dev(synth.normal_f32((n, 64), 1.0, 1)), bs)  # fp32 X
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_spmm_blocksparse(g, dev(synth.normal_bf16((n, 96), 1.0, 1)), bs)  # F % 64
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED
