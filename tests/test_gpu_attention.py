"""GPU parity of steps a3-a5 (projection, fused GATv2, fused Graph
Transformer attention on the CSR path) against the CPU oracle, through the
C ABI.  Marked gpu."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G
from tests.tolerance import TOL_BF16, TOL_F32, assert_lse_close, assert_rowwise_close

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
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def hub_graph(n, hubs, deg, seed, extra=4):
    rng = np.random.default_rng(seed)
    edges = [(int(s), h) for h in hubs for s in rng.choice(n, deg, replace=False)]
    edges += [(int(rng.integers(n)), int(rng.integers(n))) for _ in range(extra * n)]
    return G.from_edges(n, edges)


TINY = [lambda: G.random_graph(7, 0.3, 0), lambda: G.random_graph(40, 0.1, 2),
        lambda: G.star(17), lambda: G.from_edges(9, [], self_loops=False),
        lambda: G.from_edges(12, [(a, b) for a in range(12) for b in range(12)]),
        lambda: G.from_edges(5, [(0, 1)], self_loops=False)]


def check_gatv2(gnn, rp, ci, H, W, a, heads, D, slope=0.2, W_r=None, rows=None, tol=TOL_F32,
                lse_tol=1e-4):
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, lse = gnn.gnn_gatv2_fwd(g, dev(H), dev(W), dev(a), heads, D, slope,
                                 W_r=None if W_r is None else dev(W_r))
    ro, rl = oracle.gatv2(rp, ci, H, W, a, heads, D, slope, W_r=W_r, rows=rows)
    sel = slice(None) if rows is None else rows
    assert_rowwise_close(out.cpu().numpy()[sel], ro, tol, "gatv2 out")
    assert_lse_close(lse.cpu().numpy()[sel], rl, lse_tol, "gatv2 lse")


@pytest.mark.parametrize("heads,D,F_in,sep", [(1, 32, 32, False), (2, 32, 16, True),
                                              (4, 32, 64, False), (2, 64, 32, True),
                                              (1, 128, 32, False), (8, 128, 32, False)])
def test_gatv2_fp32_tiny_graphs(gnn, heads, D, F_in, sep):
    rng = np.random.default_rng(heads * 100 + D)
    HD = heads * D
    for mk in TINY:
        rp, ci = mk()
        n = len(rp) - 1
        H = rng.standard_normal((n, F_in)).astype(np.float32)
        W = (rng.standard_normal((F_in, HD)) / math.sqrt(F_in)).astype(np.float32)
        Wr = (rng.standard_normal((F_in, HD)) / math.sqrt(F_in)).astype(np.float32) if sep else None
        a = (rng.standard_normal((heads, D)) / math.sqrt(D)).astype(np.float32)
        check_gatv2(gnn, rp, ci, H, W, a, heads, D, 0.2, W_r=Wr)


def test_gatv2_heavy_rows_and_slopes(gnn):
    rp, ci = hub_graph(2000, (0, 5, 1999), 1800, 3)
    n = len(rp) - 1
    for slope, heads, D in [(0.2, 4, 32), (0.01, 2, 64), (1.0, 1, 32)]:
        HD = heads * D
        H = synth.normal_f32((n, 32), 1.0, 31)
        W = synth.normal_f32((32, HD), 1.0 / 32, 32)
        a = synth.normal_f32((heads, D), 1.0 / D, 33)
        check_gatv2(gnn, rp, ci, H, W, a, heads, D, slope)


def test_gatv2_bf16(gnn):
    rp, ci = hub_graph(3000, (1, 2000), 2600, 4)
    n = len(rp) - 1
    H = synth.normal_bf16((n, 256), 1.0, 41)
    W = synth.normal_bf16((256, 256), 1.0 / 256, 42)
    a = synth.normal_f32((4, 64), 1.0 / 64, 43)
    check_gatv2(gnn, rp, ci, H, W, a, 4, 64, tol=TOL_BF16, lse_tol=TOL_BF16)


def test_gatv2_config1(gnn):
    w = synth.workload("c1_er1k")
    check_gatv2(gnn, w["rowptr"], w["colidx"], w["X"], w["W"], w["a"], 1, 32, w["slope"])


def test_gatv2_config3_sampled(gnn):
    w = synth.workload("c3_rmat20_gatv2")
    rp, ci = w["rowptr"], w["colidx"]
    deg = np.diff(rp)
    rng = np.random.default_rng(1)
    heavy = np.argsort(-deg, kind="stable")[:2]
    cross = np.searchsorted(rp, np.arange(128, len(ci), 128 * 9973), side="right") - 1
    rows = np.unique(np.concatenate([heavy, cross[:40], rng.choice(len(deg), 150, replace=False),
                                     [0, len(deg) - 1]])).astype(np.int32)
    check_gatv2(gnn, rp, ci, w["H"], w["W"], w["a"], 4, 64, w["slope"], rows=rows,
                tol=TOL_BF16, lse_tol=TOL_BF16)


def test_gatv2_config3_error_split(gnn):
    """Splits the bf16 layer's error against the exact oracle into its two
    sources: the oracle's diagnostic mode rounds the projected features to
    bf16 as the kernel stores them, so the error left against it is the
    kernel's own arithmetic."""
    from tests.tolerance import rowwise_rel_err
    w = synth.workload("c3_rmat20_gatv2")
    rp, ci = w["rowptr"], w["colidx"]
    deg = np.diff(rp)
    rows = np.unique(np.concatenate([np.argsort(-deg, kind="stable")[:2],
                                     np.random.default_rng(4).choice(len(deg), 150, replace=False)]
                                    )).astype(np.int32)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, _ = gnn.gnn_gatv2_fwd(g, dev(w["H"]), dev(w["W"]), dev(w["a"]), 4, 64, w["slope"])
    got = out.cpu().numpy()[rows]
    exact, _ = oracle.gatv2(rp, ci, w["H"], w["W"], w["a"], 4, 64, w["slope"], rows=rows)
    rounded, _ = oracle.gatv2(rp, ci, w["H"], w["W"], w["a"], 4, 64, w["slope"], rows=rows,
                              round_c=True)
    e_exact, e_kernel, e_storage = (float(np.max(rowwise_rel_err(x, r)[0])) for x, r in
                                    ((got, exact), (got, rounded), (rounded, exact)))
    print(f"GATV2_ERROR_SPLIT total={e_exact:.3e} kernel={e_kernel:.3e} storage={e_storage:.3e}")
    assert e_exact <= TOL_BF16 and e_kernel <= TOL_BF16


def test_projection_bf16_and_fp32(gnn):
    rng = np.random.default_rng(5)
    for n, Fi, Fo in [(1000, 256, 256), (300, 64, 128), (129, 128, 64), (7, 64, 16)]:
        H = synth.normal_bf16((n, Fi), 1.0, 51)
        W = synth.normal_bf16((Fi, Fo), 1.0 / Fi, 52)
        C = gnn.gnn_projection(dev(H), dev(W)).float().cpu().numpy()
        ref = synth.bf16_to_f32(H).astype(np.float64) @ synth.bf16_to_f32(W).astype(np.float64)
        assert_rowwise_close(C, ref, 2 ** -7, f"projection bf16 {n}x{Fi}x{Fo}")
        Hf = rng.standard_normal((n, Fi)).astype(np.float32)
        Wf = rng.standard_normal((Fi, Fo)).astype(np.float32)
        Cf = gnn.gnn_projection(dev(Hf), dev(Wf)).cpu().numpy()
        assert_rowwise_close(Cf, Hf.astype(np.float64) @ Wf.astype(np.float64), TOL_F32,
                             f"projection fp32 {n}x{Fi}x{Fo}")


# ------------------------------------------------------------------ GT

def check_gt(gnn, rp, ci, Q, K, V, heads, D, scale, rows=None, tol=TOL_F32, lse_tol=1e-4):
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, lse = gnn.gnn_gt_attn_fwd(g, dev(Q), dev(K), dev(V), heads, D, scale)
    ro, rl = oracle.gt(rp, ci, Q, K, V, heads, D, scale, rows=rows)
    sel = slice(None) if rows is None else rows
    assert_rowwise_close(out.cpu().numpy()[sel], ro, tol, "gt out")
    assert_lse_close(lse.cpu().numpy()[sel], rl, lse_tol, "gt lse")


@pytest.mark.parametrize("heads,D", [(1, 32), (2, 32), (8, 32), (2, 64), (4, 128)])
def test_gt_fp32_tiny_graphs(gnn, heads, D):
    rng = np.random.default_rng(heads * 7 + D)
    for mk in TINY:
        rp, ci = mk()
        n = len(rp) - 1
        Q, K, V = (rng.standard_normal((n, heads * D)).astype(np.float32) for _ in range(3))
        check_gt(gnn, rp, ci, Q, K, V, heads, D, 1.0 / math.sqrt(D))


def test_gt_heavy_rows_fp32_and_bf16(gnn):
    rp, ci = hub_graph(2500, (3, 1200), 2200, 6)
    n = len(rp) - 1
    Q, K, V = (synth.normal_f32((n, 256), 1.0, 60 + k) for k in range(3))
    check_gt(gnn, rp, ci, Q, K, V, 8, 32, 1.0 / math.sqrt(32))
    Qb, Kb, Vb = (synth.normal_bf16((n, 256), 1.0, 70 + k) for k in range(3))
    check_gt(gnn, rp, ci, Qb, Kb, Vb, 8, 32, 1.0 / math.sqrt(32), tol=TOL_BF16, lse_tol=TOL_BF16)


def test_gt_config4_sampled(gnn):
    w = synth.workload("c4_clustered_gt")
    rp, ci = w["rowptr"], w["colidx"]
    deg = np.diff(rp)
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([np.argsort(-deg, kind="stable")[:8],
                                     rng.choice(len(deg), 300, replace=False),
                                     [0, len(deg) - 1]])).astype(np.int32)
    check_gt(gnn, rp, ci, w["Q"], w["K"], w["V"], 8, 32, w["scale"], rows=rows, tol=TOL_BF16,
             lse_tol=TOL_BF16)


# ------------------------------------------------------- GT, tensor-core tiles

def clustered_small(n_clusters, size=256, p=0.3, seed=2, n_extra=None):
    rng = np.random.default_rng(seed)
    edges = []
    for c in range(n_clusters):
        base = c * size
        m = rng.random((size, size)) < p
        d, s = np.nonzero(m)
        edges += [(base + int(b), base + int(a)) for a, b in zip(d, s)]
    n = n_clusters * size
    for _ in range(n // 2 if n_extra is None else n_extra):
        edges.append((int(rng.integers(n)), int(rng.integers(n))))
    return G.from_edges(n, edges)


def check_gt_tiles(gnn, rp, ci, Q, K, V, heads, D, scale, thr, rows=None, packing=0):
    g = gnn.graph_prepare(dev(rp), dev(ci))
    bs = gnn.gnn_blocksparse_build(g, thr, packing=packing)
    out, lse = gnn.gnn_gt_attn_fwd(g, dev(Q), dev(K), dev(V), heads, D, scale, bs=bs)
    ro, rl = oracle.gt(rp, ci, Q, K, V, heads, D, scale, rows=rows)
    sel = slice(None) if rows is None else rows
    assert_rowwise_close(out.cpu().numpy()[sel], ro, TOL_BF16, f"gt tiles out thr={thr}")
    assert_lse_close(lse.cpu().numpy()[sel], rl, TOL_BF16, f"gt tiles lse thr={thr}")
    return bs


@pytest.mark.parametrize("thr", [0.0, 0.25, 0.35, 1.0])
@pytest.mark.parametrize("heads,D", [(8, 32), (2, 64)])
def test_gt_tiles_small_clustered(gnn, thr, heads, D):
    # 5 clusters of 256 nodes (10 row groups, one of them ragged by the extra
    # 40 nodes), cross-cluster edges that land in sparse tiles
    rp, ci = clustered_small(5, p=0.3, seed=heads)
    n = len(rp) - 1
    Q, K, V = (synth.normal_bf16((n, heads * D), 1.0, 80 + k) for k in range(3))
    check_gt_tiles(gnn, rp, ci, Q, K, V, heads, D, 1.0 / math.sqrt(D), thr)


def test_gt_tiles_ragged_group_and_dense_block(gnn):
    # 300 nodes: the last 128-row group is partial; a 60-node clique gives
    # full tiles, a sparse rest gives residual edges
    rp, ci = G.from_edges(300, [(a, b) for a in range(60) for b in range(60)] +
                          [(i, (7 * i + 3) % 300) for i in range(300)])
    n = len(rp) - 1
    Q, K, V = (synth.normal_bf16((n, 256), 1.0, 90 + k) for k in range(3))
    for thr in (0.0, 0.5):
        check_gt_tiles(gnn, rp, ci, Q, K, V, 8, 32, 1.0 / math.sqrt(32), thr)


@pytest.mark.parametrize("D", [32, 64])
def test_gt_tiles_empty_groups_and_rows_without_residual(gnn, D):
    """Every edge in a tile (threshold 0), so the tile kernel writes all rows
    itself: row groups 1 and 3 (rows 128..255, 384..511) have no edges at
    all, and single rows inside tiled groups have none either; they must come
    out as 0 with lse = -inf."""
    n = 600
    rng = np.random.default_rng(11)
    empty = set(range(128, 256)) | set(range(384, 512)) | {5, 70, 300, 599}
    edges = [(int(rng.integers(n)), d) for d in range(n) if d not in empty for _ in range(6)]
    rp, ci = G.from_edges(n, edges, self_loops=False)
    assert all(rp[r + 1] == rp[r] for r in empty)
    heads = 256 // D
    Q, K, V = (synth.normal_bf16((n, 256), 1.0, 95 + k) for k in range(3))
    bs = check_gt_tiles(gnn, rp, ci, Q, K, V, heads, D, 1.0 / math.sqrt(D), 0.0)
    assert bs.meta.nnz_residual == 0 and bs.meta.n_tiles_kept > 0


def test_gt_tiles_config4_sampled(gnn):
    w = synth.workload("c4_clustered_gt")
    rp, ci = w["rowptr"], w["colidx"]
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(len(rp) - 1, 300, replace=False),
                                     [0, 127, 128, len(rp) - 2]])).astype(np.int32)
    # every fill threshold the benchmark reports on this graph
    for thr in (0.0, 0.1, 0.2, 0.3, 0.5):
        bs = check_gt_tiles(gnn, rp, ci, w["Q"], w["K"], w["V"], 8, 32, w["scale"], thr, rows=rows)
        if thr == 0.0:
            assert bs.meta.nnz_residual == 0 and bs.meta.n_tiles_kept > 0
    # columns in count-sorted order (the tile kernels take any column order)
    for thr in (0.0, 0.3):
        check_gt_tiles(gnn, rp, ci, w["Q"], w["K"], w["V"], 8, 32, w["scale"], thr, rows=rows,
                       packing=1)


@pytest.mark.parametrize("D", [32, 64])
def test_gt_tiles_count_packing_small_clustered(gnn, D):
    rp, ci = clustered_small(3, p=0.3, seed=D)
    n = len(rp) - 1
    heads = 256 // D
    Q, K, V = (synth.normal_bf16((n, 256), 1.0, 85 + k) for k in range(3))
    for thr in (0.0, 0.3, 0.4):
        check_gt_tiles(gnn, rp, ci, Q, K, V, heads, D, 1.0 / math.sqrt(D), thr, packing=1)
