"""GPU parity of step a6 (16x16 block-sparse tile layout) against the CPU
oracle, through the C ABI: every array and count is compared bit-exactly.
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


def check(gnn, rp, ci, thr, packing=0):
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    bs = gnn.gnn_blocksparse_build(g, thr, packing=packing)
    assert bs.meta.packing == packing
    ref = oracle.blocksparse(rp, ci, thr, packing=packing)
    m = bs.meta
    assert (m.n_blocks, m.n_tiles_kept, m.nnz_tiles, m.nnz_residual) == \
        (ref["n_blocks"], ref["n_tiles_kept"], ref["nnz_tiles"], ref["nnz_residual"]), thr
    got = {k: v.cpu().numpy() for k, v in bs.arrays().items()}
    assert np.array_equal(got["grp_blk_offset"], ref["grp_blk_offset"])
    assert np.array_equal(got["blk_cols"], ref["blk_cols"])
    assert np.array_equal(got["blk_mask"].view(np.uint64), ref["blk_mask"])
    assert np.array_equal(got["res_rowptr"], ref["res_rowptr"])
    assert np.array_equal(got["res_colidx"], ref["res_colidx"])
    return bs


def clustered_small(n_clusters=6, size=256, p=0.3, seed=2):
    rng = np.random.default_rng(seed)
    edges = []
    for c in range(n_clusters):
        base = c * size
        m = rng.random((size, size)) < p
        d, s = np.nonzero(m)
        edges += [(base + int(a), base + int(b)) for b, a in zip(d, s)]
    for _ in range(n_clusters * size // 2):
        edges.append((int(rng.integers(n_clusters * size)), int(rng.integers(n_clusters * size))))
    return G.from_edges(n_clusters * size, edges)


@pytest.mark.parametrize("packing", [0, 1])
@pytest.mark.parametrize("thr", [0.0, 0.02, 0.1, 0.3, 0.5, 1.0])
def test_blocksparse_small_graphs(gnn, thr, packing):
    for rp, ci in (G.random_graph(40, 0.1, 1), G.from_edges(300, [(a, b) for a in range(60) for b in range(60)]),
                   G.star(150), G.from_edges(10, [], self_loops=False), clustered_small()):
        check(gnn, rp, ci, thr, packing)


def test_blocksparse_count_packing_config4(gnn):
    """Count-sorted packing (columns by descending edge count in the group,
    ties by id) on the clustered graph, bit for bit, at the fills where it
    changes which tiles are kept."""
    w = synth.workload("c4_clustered_gt", features=False)
    kept = {}
    for thr in (0.0, 0.3, 0.4, 0.5):
        bs = check(gnn, w["rowptr"], w["colidx"], thr, packing=1)
        assert bs.meta.nnz_tiles + bs.meta.nnz_residual == len(w["colidx"])
        kept[thr] = bs.meta.n_tiles_kept
    assert kept[0.0] >= kept[0.3] >= kept[0.4] >= kept[0.5]


def test_blocksparse_rejects_unknown_packing(gnn):
    import ctypes
    rp, ci = G.random_graph(40, 0.1, 1)
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    ws = g.workspace(gnn.GNN_OP_BLOCKSPARSE)
    meta = gnn.binding.gnn_blocksparse()
    nbytes = ctypes.c_size_t(0)
    rc = gnn.lib().gnn_blocksparse_plan_packed(ctypes.byref(g.csr), 0.0, 2, ws.data_ptr(),
                                               ws.numel(), ctypes.byref(meta),
                                               ctypes.byref(nbytes), None)
    assert rc == gnn.GNN_ERR_INVALID_ARG


def test_blocksparse_config4_both_thresholds(gnn):
    w = synth.workload("c4_clustered_gt", features=False)
    for thr in (0.5, 0.0):
        bs = check(gnn, w["rowptr"], w["colidx"], thr)
        assert bs.meta.nnz_tiles + bs.meta.nnz_residual == len(w["colidx"])


def test_blocksparse_rejects_a_plan_of_another_graph(gnn):
    """A plan made for one graph is refused for another, and nothing is
    written: a layout that would not fit the buffer (workspace error), or
    counts that differ from the plan's (invalid argument)."""
    import ctypes
    rp, ci = clustered_small(2)
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    bs = gnn.gnn_blocksparse_build(g, 0.0)
    before = bs.buf.clone()
    for other, expect in ((clustered_small(3, seed=5), gnn.GNN_ERR_WORKSPACE),
                          (clustered_small(2, p=0.2, seed=5), gnn.GNN_ERR_INVALID_ARG)):
        g2 = gnn.Graph(dev(other[0]), dev(other[1]), prepare=False)
        meta = gnn.binding.gnn_blocksparse()
        ctypes.pointer(meta)[0] = bs.meta
        meta.n_rows = g2.n_rows
        ws = g2.workspace(gnn.GNN_OP_BLOCKSPARSE)
        rc = gnn.lib().gnn_blocksparse_build(ctypes.byref(g2.csr), ctypes.byref(meta),
                                             bs.buf.data_ptr(), bs.buf.numel(), ws.data_ptr(),
                                             ws.numel(), None)
        assert rc == expect
        torch.cuda.synchronize()
        assert torch.equal(bs.buf, before)
