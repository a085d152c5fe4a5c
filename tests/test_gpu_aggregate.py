"""GPU parity of steps a0-a2 (prep, SpMM, segment sum/mean/max) against the
CPU oracle, through the C ABI.  Marked gpu."""
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


def feats_to_dev(X):
    """numpy fp32 or bf16 bits (uint16) -> CUDA tensor of the same dtype."""
    if X.dtype == np.uint16:
        return dev(X.view(np.int16)).view(torch.bfloat16)
    return dev(X)


def check_exact_max(y, am, ref_y, ref_am):
    """max or min: values bit for bit (signed zeros included), arg exactly"""
    ref32 = ref_y.astype(np.float32)
    assert np.array_equal(y.view(np.uint32), ref32.view(np.uint32)), "max/min values differ"
    assert np.array_equal(am, ref_am), "argmax/argmin differs"


def run_all(gnn, rp, ci, X, rows=None, tol=TOL_F32, mappings=(0, 1, 2), norms=(0, 1, 2, 3),
            values=None):
    g = gnn.graph_prepare(dev(rp), dev(ci), None if values is None else dev(values))
    Xd = feats_to_dev(X)
    sel = slice(None) if rows is None else rows
    for norm in norms:
        ref = oracle.spmm(rp, ci, X, norm=norm, values=values, rows=rows)
        for mp in mappings:
            Y = gnn.gnn_spmm(g, Xd, norm=norm, mapping=mp).cpu().numpy()
            assert_rowwise_close(Y[sel], ref, tol, f"spmm norm={norm} map={mp}")
    if values is not None:
        return
    ys = gnn.gnn_segment_reduce_sum(g, Xd).cpu().numpy()
    assert_rowwise_close(ys[sel], oracle.segment_reduce(oracle.OP_SUM, rp, ci, X, rows=rows), tol,
                         "sum")
    ym = gnn.gnn_segment_reduce_mean(g, Xd).cpu().numpy()
    assert_rowwise_close(ym[sel], oracle.segment_reduce(oracle.OP_MEAN, rp, ci, X, rows=rows), tol,
                         "mean")
    yx, am = gnn.gnn_segment_reduce_max(g, Xd)
    ry, ram = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X, rows=rows)
    check_exact_max(yx.cpu().numpy()[sel], am.cpu().numpy()[sel], ry, ram)
    yn, an = gnn.gnn_segment_reduce_min(g, Xd)
    rn, ran = oracle.segment_reduce(oracle.OP_MIN, rp, ci, X, rows=rows)
    check_exact_max(yn.cpu().numpy()[sel], an.cpu().numpy()[sel], rn, ran)
    return g


def _hub_graph(n=3000, hubs=(0, 17, 2999), deg=2500, seed=0):
    rng = np.random.default_rng(seed)
    edges = [(int(s), h) for h in hubs for s in rng.choice(n, deg, replace=False)]
    edges += [(int(rng.integers(n)), int(rng.integers(n))) for _ in range(4 * n)]
    return G.from_edges(n, edges)


@pytest.mark.parametrize("F", [32, 64, 128, 256])
def test_tiny_graphs_fp32(gnn, F):
    rng = np.random.default_rng(F)
    for k, (rp, ci) in enumerate([G.random_graph(7, 0.3, 0), G.random_graph(40, 0.1, 2, False),
                                  G.star(17), G.from_edges(9, [], self_loops=False),
                                  G.from_edges(12, [(a, b) for a in range(12) for b in range(12)]),
                                  G.from_edges(5, [(0, 1)], self_loops=False)]):
        n = len(rp) - 1
        X = rng.standard_normal((n, F)).astype(np.float32)
        run_all(gnn, rp, ci, X)


def test_ties_and_signed_zero_max_exact(gnn):
    rng = np.random.default_rng(3)
    rp, ci = _hub_graph(600, hubs=(5, 300), deg=550)
    X = rng.integers(-3, 4, (600, 32)).astype(np.float32)
    X[rng.random(X.shape) < 0.2] = -0.0
    g = gnn.graph_prepare(dev(rp), dev(ci))
    yx, am = gnn.gnn_segment_reduce_max(g, dev(X))
    ry, ram = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
    check_exact_max(yx.cpu().numpy(), am.cpu().numpy(), ry, ram)


def test_min_ties_and_signed_zero_exact(gnn):
    rng = np.random.default_rng(4)
    for F in (32, 128):  # k_agg_auto and the edge-span kernel
        rp, ci = _hub_graph(600, hubs=(5, 300), deg=550)
        X = rng.integers(-3, 4, (600, F)).astype(np.float32)
        X[rng.random(X.shape) < 0.2] = -0.0
        g = gnn.graph_prepare(dev(rp), dev(ci))
        yn, an = gnn.gnn_segment_reduce_min(g, dev(X))
        rn, ran = oracle.segment_reduce(oracle.OP_MIN, rp, ci, X)
        check_exact_max(yn.cpu().numpy(), an.cpu().numpy(), rn, ran)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_heavy_rows_split_across_workers(gnn, dtype):
    rp, ci = _hub_graph()
    n = len(rp) - 1
    if dtype == "f32":
        X, tol = synth.normal_f32((n, 128), 1.0, 11), TOL_F32
    else:
        X, tol = synth.normal_bf16((n, 256), 1.0, 11), TOL_BF16
    run_all(gnn, rp, ci, X, tol=tol)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_heavy_rows_on_sub_warp_workers(gnn, dtype):
    """Rows of 8 chunks (F = 32 fp32, F = 64 bf16) run on 8-lane workers, four
    to a warp, each over its own run of edges (the slice-coalescing mapping
    for small F); hub rows of degree 2500 are cut across ~40 runs and their
    pieces merged."""
    rp, ci = _hub_graph(seed=5)
    n = len(rp) - 1
    if dtype == "f32":
        X, tol = synth.normal_f32((n, 32), 1.0, 13), TOL_F32
    else:
        X, tol = synth.normal_bf16((n, 64), 1.0, 13), TOL_BF16
    run_all(gnn, rp, ci, X, tol=tol, mappings=(0,))


def test_edge_values_and_wide_features(gnn):
    rp, ci = _hub_graph(1500, hubs=(3,), deg=1400, seed=4)
    n = len(rp) - 1
    vals = synth.uniform_f32(len(ci), 0.5, 2.0, 9)
    X = synth.normal_f32((n, 512), 1.0, 12)
    run_all(gnn, rp, ci, X, values=vals)
    run_all(gnn, rp, ci, X, mappings=(0,), norms=(3,))


def test_empty_graph_and_trailing_empty_rows(gnn):
    X = np.ones((10, 32), np.float32)
    run_all(gnn, *G.from_edges(10, [], self_loops=False), X)
    rp, ci = G.from_edges(300, [(i, 3) for i in range(1, 290)], self_loops=False)
    run_all(gnn, rp, ci, np.random.default_rng(0).standard_normal((300, 32)).astype(np.float32))


def _short_rows_graph(n=6000, seed=7):
    """Rows of degree 0, 1 and 2 in random order (so one 64-edge span holds
    more than 32 rows), a run of 700 empty rows, 300 trailing empty rows and
    two heavy rows."""
    rng = np.random.default_rng(seed)
    deg = rng.choice([0, 1, 1, 2], n)
    deg[2000:2700] = 0
    deg[n - 300:] = 0
    deg[[100, 4000]] = [900, 2100]
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    ci = np.concatenate([np.sort(rng.choice(n, d, replace=False)) for d in deg]).astype(np.int32)
    return rp, ci


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_rows_and_empty_runs(gnn, dtype):
    rp, ci = _short_rows_graph()
    n = len(rp) - 1
    if dtype == "f32":
        X, tol = synth.normal_f32((n, 128), 1.0, 21), TOL_F32
    else:
        X, tol = synth.normal_bf16((n, 256), 1.0, 21), TOL_BF16
    run_all(gnn, rp, ci, X, tol=tol)


def test_unprepared_graph(gnn):
    """Without the prepared graph each run finds its rows by search."""
    rp, ci = _hub_graph(2000, hubs=(1, 1999), deg=1500, seed=6)
    n = len(rp) - 1
    X = synth.normal_f32((n, 128), 1.0, 13)
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    Xd = dev(X)
    assert_rowwise_close(gnn.gnn_spmm(g, Xd, norm=gnn.GNN_NORM_NONE).cpu().numpy(),
                         oracle.spmm(rp, ci, X, norm=oracle.NORM_NONE), TOL_F32, "spmm, no prep")
    assert_rowwise_close(gnn.gnn_segment_reduce_sum(g, Xd).cpu().numpy(),
                         oracle.segment_reduce(oracle.OP_SUM, rp, ci, X), TOL_F32, "sum, no prep")
    assert_rowwise_close(gnn.gnn_segment_reduce_mean(g, Xd).cpu().numpy(),
                         oracle.segment_reduce(oracle.OP_MEAN, rp, ci, X), TOL_F32, "mean, no prep")
    yx, am = gnn.gnn_segment_reduce_max(g, Xd)
    ry, ram = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
    check_exact_max(yx.cpu().numpy(), am.cpu().numpy(), ry, ram)
    yn, an = gnn.gnn_segment_reduce_min(g, Xd)
    rn, ran = oracle.segment_reduce(oracle.OP_MIN, rp, ci, X)
    check_exact_max(yn.cpu().numpy(), an.cpu().numpy(), rn, ran)


@pytest.mark.parametrize("op", ["max", "min"])
def test_reduce_backward_config2(gnn, op):
    """grad_X of max / min from the oracle's own arg (every row of R-MAT
    scale 17, F = 128) and a random output gradient."""
    w = synth.workload("c2_rmat17")
    rp, ci, X = w["rowptr"], w["colidx"], w["X"]
    code = oracle.OP_MAX if op == "max" else oracle.OP_MIN
    _, arg = oracle.segment_reduce(code, rp, ci, X)
    go = synth.normal_f32(arg.shape, 1.0, 51)
    n = len(rp) - 1
    gx = gnn.gnn_segment_reduce_ext_backward(dev(arg), dev(go), n).cpu().numpy()
    assert_rowwise_close(gx, oracle.reduce_ext_backward(arg, go.astype(np.float64), n), TOL_F32,
                         f"{op} backward")


def test_reduce_backward_shared_sources_and_bad_index(gnn):
    arg = np.array([[2, -1, 2, 0], [2, 0, -1, 0], [-1, 0, 1, 1]], np.int32)
    go = np.arange(12, dtype=np.float32).reshape(3, 4) + 1
    gx = gnn.gnn_segment_reduce_ext_backward(dev(arg), dev(go), 3).cpu().numpy()
    assert np.array_equal(gx, oracle.reduce_ext_backward(arg, go.astype(np.float64), 3))
    # an index past n_cols is caught by the kernel's bounds check and reported
    gnn.gnn_segment_reduce_ext_backward(dev(np.array([[0, 0, 0, 9]], np.int32)),
                                        dev(np.ones((1, 4), np.float32)), 3)
    assert gnn.last_device_error() == gnn.GNN_ERR_DEVICE_CHECK
    assert gnn.last_device_error() == 0


def test_config1_er(gnn):
    w = synth.workload("c1_er1k")
    run_all(gnn, w["rowptr"], w["colidx"], w["X"])


def test_config2_rmat17_sampled(gnn):
    w = synth.workload("c2_rmat17")
    rp, ci, X = w["rowptr"], w["colidx"], w["X"]
    deg = np.diff(rp)
    rng = np.random.default_rng(0)
    # the heaviest rows, rows whose edges cross run boundaries, random rows
    heavy = np.argsort(-deg, kind="stable")[:24]
    bnd = np.searchsorted(rp, np.arange(256, len(ci), 256 * 97), side="right") - 1
    rows = np.unique(np.concatenate([heavy, bnd, rng.choice(len(deg), 400, replace=False),
                                     [0, len(deg) - 1]])).astype(np.int32)
    run_all(gnn, rp, ci, X, rows=rows)


@pytest.mark.parametrize("graph", ["rmat19_ef20", "c3_rmat20"])
def test_longer_spans_on_larger_graphs(gnn, graph):
    """Graphs of 2^23..2^24 edges run 128-edge spans and larger ones 256-edge
    spans; SpMM (all norms and mappings), sum, mean and max on sampled rows
    (the heaviest, rows around span boundaries, random rows)."""
    if graph == "rmat19_ef20":
        rp, ci = synth.rmat(19, 20)
        assert (1 << 23) <= len(ci) < (1 << 24)
    else:
        w = synth.workload("c3_rmat20_gatv2", features=False)
        rp, ci = w["rowptr"], w["colidx"]
        assert len(ci) >= (1 << 24)
    n = len(rp) - 1
    X = synth.normal_f32((n, 128), 1.0, 31)
    deg = np.diff(rp)
    rng = np.random.default_rng(7)
    span = 128 if len(ci) < (1 << 24) else 256
    bnd = np.searchsorted(rp, np.arange(span, len(ci), span * 1013), side="right") - 1
    rows = np.unique(np.concatenate([np.argsort(-deg, kind="stable")[:8], bnd,
                                     rng.choice(n, 150, replace=False), [0, n - 1]])).astype(np.int32)
    run_all(gnn, rp, ci, X, rows=rows, norms=(0, 3))


def test_repeat_calls_reuse_the_workspace(gnn):
    # with the prepared graph, heavy-row pieces are summed in edge order, so
    # repeats are bit-identical; max is exact in any order.  Both show that
    # the workspace slots and tickets are left ready for the next call.
    w = synth.workload("c2_rmat17")
    g = gnn.graph_prepare(dev(w["rowptr"]), dev(w["colidx"]))
    Xd = dev(w["X"])
    a = gnn.gnn_spmm(g, Xd)
    b = gnn.gnn_spmm(g, Xd)
    assert torch.equal(a, b), "spmm repeat differs"
    s1 = gnn.gnn_segment_reduce_sum(g, Xd)
    s2 = gnn.gnn_segment_reduce_sum(g, Xd)
    assert torch.equal(s1, s2), "sum repeat differs"
    m1, i1 = gnn.gnn_segment_reduce_max(g, Xd)
    m2, i2 = gnn.gnn_segment_reduce_max(g, Xd)
    assert torch.equal(m1, m2) and torch.equal(i1, i2)
    # without the prepared graph pieces are folded by fp32 atomics: equal to rounding
    g0 = gnn.Graph(dev(w["rowptr"]), dev(w["colidx"]), prepare=False)
    c = gnn.gnn_segment_reduce_sum(g0, Xd).cpu().numpy()
    assert_rowwise_close(c, s1.cpu().numpy(), 1e-6, "sum without prep")


def test_validate_flags_bad_csr(gnn):
    rp = np.array([0, 2, 3], np.int32)
    ci = np.array([1, 0, 5], np.int32)  # column 5 out of range, row 0 unsorted
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    assert gnn.csr_validate(g) == gnn.GNN_ERR_DEVICE_CHECK
    rp2, ci2 = G.random_graph(30, 0.2, 1)
    assert gnn.csr_validate(gnn.Graph(dev(rp2), dev(ci2), prepare=False)) == 0


def test_host_validation_rejects_bad_arguments(gnn):
    rp, ci = G.random_graph(30, 0.2, 1)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_spmm(g, dev(np.ones((30, 12), np.float32)))      # F=12: 3 chunks
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED
    X = torch.ones(30 * 32 + 1, device="cuda")[1:].view(30, 32)  # misaligned rows
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_segment_reduce_sum(g, X)
    assert e.value.code == gnn.GNN_ERR_INVALID_ARG


def test_config5_rmat22_sampled_original_and_degree_order(gnn):
    """GCN SpMM at full size (R-MAT scale 22, X bf16 [N,256]) in the launch
    configuration the benchmark times, on sampled rows, with the original ids
    and after a degree-order relabel done on the GPU."""
    w = synth.workload("c5_rmat22")
    rp, ci, X = w["rowptr"], w["colidx"], w["X"]
    deg = np.diff(rp)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([np.argsort(-deg, kind="stable")[:3],
                                     rng.choice(len(deg), 200, replace=False),
                                     [0, len(deg) - 1]])).astype(np.int32)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    Xd = feats_to_dev(X)
    Y = gnn.gnn_spmm(g, Xd, norm=gnn.GNN_NORM_BOTH).cpu().numpy()
    assert_rowwise_close(Y[rows], oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH, rows=rows),
                         TOL_BF16, "c5 spmm")
    perm, inv = gnn.gnn_reorder_perm(g, gnn.GNN_PERM_DEGREE)
    rp2, ci2, X2 = gnn.gnn_apply_perm(g, perm, inv, X=Xd)
    g2 = gnn.graph_prepare(rp2, ci2)
    Y2 = gnn.gnn_spmm(g2, X2, norm=gnn.GNN_NORM_BOTH).cpu().numpy()
    p = perm.cpu().numpy()
    inv_h = inv.cpu().numpy()
    # row r of the relabelled result is row p[r] of the original one
    assert_rowwise_close(Y2[inv_h[rows]], oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH, rows=rows),
                         TOL_BF16, "c5 spmm, degree order")
    assert np.array_equal(p[inv_h[rows]], rows)
