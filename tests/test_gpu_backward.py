"""GPU parity of the CSR^T build, of the SpMM backward run as a SpMM on
CSR^T, and of the Graph Transformer and GATv2 attention backward passes,
against the CPU oracle, through the C ABI.  Marked gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G
from tests.tolerance import TOL_BF16, TOL_F32, assert_rowwise_close, assert_terms_close

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


def test_gt_backward_rmat_power_law(gnn):
    """R-MAT scale 13 (8,192 nodes, ~130K edges): power-law rows from one
    edge to hundreds, so hub destinations (dQ over the CSR) and hub sources
    (dK, dV over CSR^T) are both exercised."""
    rp, ci = synth.rmat(13, 16)
    assert np.max(np.diff(rp)) > 300
    check_gt_backward(gnn, rp, ci, 8, 32, seed=3)


def test_gt_backward_clustered(gnn):
    rp, ci = synth.clustered(32, 128, 0.3, 0.02, 5)
    check_gt_backward(gnn, rp, ci, 8, 32, seed=1)


def test_gt_backward_config4_sampled(gnn):
    """The clustered 262K-node graph, 8 heads x 32, bf16 (the shape the
    backward is timed on), on sampled outputs the oracle computes exactly:
    dQ of a row needs only its own edge list; dK and dV of a source need
    every row that lists it, each whole."""
    w = synth.workload("c4_clustered_gt", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n, heads, D = len(rp) - 1, 8, 32
    scale = 1.0 / np.sqrt(D)
    Q, K, V = (_bf16((n, heads * D), 170 + k) for k in range(3))
    dO = synth.normal_f32((n, heads * D), 1.0, 180)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    qd, kd, vd = (dev(x.view(np.int16)).view(torch.bfloat16) for x in (Q, K, V))
    out, lse = gnn.gnn_gt_attn_fwd(g, qd, kd, vd, heads, D, scale)
    gt = _transpose_graph(gnn, rp, ci)
    dQ, dK, dV = (t.cpu().numpy() for t in gnn.gnn_gt_attn_bwd(g, gt, qd, kd, vd, heads, D, scale,
                                                                 out, lse, dev(dO)))
    rng = np.random.default_rng(11)
    rows = np.unique(rng.choice(n, 200, replace=False))
    srp, sci, nodes = _subgraph(rp, ci, rows)
    rQ, _, _ = oracle.gt_backward(srp, sci, Q[nodes], K[nodes], V[nodes], heads, D, scale, dO[nodes])
    assert_rowwise_close(dQ[rows], rQ[np.searchsorted(nodes, rows)], TOL_BF16, "c4 dQ")
    rpt, cit, _ = oracle.csr_transpose(rp, ci)
    js = np.unique(rng.choice(n, 40, replace=False))
    lister = np.unique(np.concatenate([cit[rpt[j]:rpt[j + 1]] for j in js]))
    srp, sci, nodes = _subgraph(rp, ci, lister)
    _, rK, rV = oracle.gt_backward(srp, sci, Q[nodes], K[nodes], V[nodes], heads, D, scale, dO[nodes])
    pos = np.searchsorted(nodes, js)
    assert_rowwise_close(dK[js], rK[pos], TOL_BF16, "c4 dK")
    assert_rowwise_close(dV[js], rV[pos], TOL_BF16, "c4 dV")


def test_gt_backward_rmat20_sampled(gnn):
    """R-MAT scale 20 (1,048,576 nodes, 17.1M edges, rows up to ~40K edges),
    8 heads x 32, bf16: the edge-run schedule the mean degree selects on
    power-law graphs (hub rows cut into 256-edge pieces summed in edge
    order), on sampled outputs the oracle computes exactly -- dQ of the
    heaviest rows and of random rows, dK and dV of the heaviest source and of
    random sources."""
    w = synth.workload("c3_rmat20_gatv2", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n, heads, D = len(rp) - 1, 8, 32
    assert len(ci) < 32 * n
    scale = 1.0 / np.sqrt(D)
    Q, K, V = (_bf16((n, heads * D), 270 + k) for k in range(3))
    dO = synth.normal_f32((n, heads * D), 1.0, 280)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    qd, kd, vd = (dev(x.view(np.int16)).view(torch.bfloat16) for x in (Q, K, V))
    out, lse = gnn.gnn_gt_attn_fwd(g, qd, kd, vd, heads, D, scale)
    gt = _transpose_graph(gnn, rp, ci)
    dQ, dK, dV = (t.cpu().numpy() for t in gnn.gnn_gt_attn_bwd(g, gt, qd, kd, vd, heads, D, scale,
                                                                 out, lse, dev(dO)))
    rng = np.random.default_rng(13)
    deg = np.diff(rp)
    rows = np.unique(np.concatenate([np.argsort(-deg, kind="stable")[:3],
                                     rng.choice(n, 150, replace=False)]))
    srp, sci, nodes = _subgraph(rp, ci, rows)
    rQ, _, _ = oracle.gt_backward(srp, sci, Q[nodes], K[nodes], V[nodes], heads, D, scale, dO[nodes])
    assert_rowwise_close(dQ[rows], rQ[np.searchsorted(nodes, rows)], TOL_BF16, "rmat20 dQ")
    rpt, cit, _ = oracle.csr_transpose(rp, ci)
    dout_t = np.diff(rpt)
    js = np.unique(np.concatenate([np.argsort(-dout_t, kind="stable")[:1],
                                   rng.choice(n, 30, replace=False)]))
    lister = np.unique(np.concatenate([cit[rpt[j]:rpt[j + 1]] for j in js]))
    srp, sci, nodes = _subgraph(rp, ci, lister)
    _, rK, rV = oracle.gt_backward(srp, sci, Q[nodes], K[nodes], V[nodes], heads, D, scale, dO[nodes])
    pos = np.searchsorted(nodes, js)
    assert_rowwise_close(dK[js], rK[pos], TOL_BF16, "rmat20 dK")
    assert_rowwise_close(dV[js], rV[pos], TOL_BF16, "rmat20 dV")


def test_gt_backward_rejects_unsupported_shapes(gnn):
    rp, ci = G.random_graph(20, 0.2, 1)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    gt = gnn.Graph(*gnn.gnn_csr_transpose(g)[:2], None, None, False)
    x = torch.zeros((20, 96), dtype=torch.bfloat16, device="cuda")
    f = torch.zeros((20, 96), dtype=torch.float32, device="cuda")
    with pytest.raises(gnn.GnnError) as e:
        gnn.gnn_gt_attn_bwd(g, gt, x, x, x, 3, 32, 0.2, f, torch.zeros((20, 3), device="cuda"), f)
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED


# ---------------------------------------------------------------- GATv2 backward

def _bf16_exact(x):
    """bf16 bit patterns of values bf16 holds exactly (0 and 1 here)."""
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _dev_feat(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def _gatv2_inputs(n, heads, D, bf16, shared, seed):
    HD = heads * D
    mk = synth.normal_bf16 if bf16 else synth.normal_f32
    Cl = mk((n, HD), 1.0, 90 + seed)
    Cr = None if shared else mk((n, HD), 1.0, 91 + seed)
    a = synth.normal_f32((heads, D), 0.25, 92 + seed)
    dO = synth.normal_f32((n, HD), 1.0, 93 + seed)
    return Cl, Cr, a, dO


def _gatv2_forward_exact(gnn, g, Cl, Cr, a, heads, D, slope):
    """The GPU forward scoring exactly Cl and Cr: H = Cl with W = I, or
    H = [Cl | Cr] with W_l = [I; 0], W_r = [0; I] (a product with 1 and sums
    with 0 are exact, so the projected rows are the given ones)."""
    HD = heads * D
    conv = _bf16_exact if Cl.dtype == np.uint16 else (lambda x: x.astype(np.float32))
    eye, zero = np.eye(HD, dtype=np.float32), np.zeros((HD, HD), np.float32)
    if Cr is None:
        return gnn.gnn_gatv2_fwd(g, _dev_feat(Cl), _dev_feat(conv(eye)), dev(a), heads, D, slope)
    H = np.hstack([Cl, Cr])
    return gnn.gnn_gatv2_fwd(g, _dev_feat(H), _dev_feat(conv(np.vstack([eye, zero]))), dev(a), heads,
                             D, slope, W_r=_dev_feat(conv(np.vstack([zero, eye]))))


def _transpose_graph(gnn, rp, ci):
    rpt, cit, _ = gnn.gnn_csr_transpose(gnn.Graph(dev(rp), dev(ci), None, None, False))
    return gnn.Graph(rpt, cit, None, None, False)


def _widen(x):
    return synth.bf16_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


def gatv2_term_scales(rp, ci, Cl, Cr, a, heads, D, dO, slope=0.2, chunk=8192):
    """Summed magnitude of the terms of dl, dr and da (shapes [n, HD], [n, HD],
    [heads, D]): a bound for the error scale, not an expected value.  A score
    gradient de_ij = alpha_ij (<dO_i, r_j> - G_i) is bounded by alpha_ij
    (P_ij + Gabs_i) with P_ij = sum_d |dO_id| |r_jd| and Gabs_i = sum_j
    alpha_ij P_ij (the same bound covers an error in the stored O that G is
    formed from), and |sigma'| <= 1, |sigma(x)| <= |x|."""
    n = len(rp) - 1
    HD = heads * D
    L = _widen(Cl).reshape(n, heads, D)
    R = L if Cr is None else _widen(Cr).reshape(n, heads, D)
    g = np.abs(np.asarray(dO, np.float64)).reshape(n, heads, D)
    av = np.asarray(a, np.float64).reshape(heads, D)
    aa = np.abs(av)
    deg = np.diff(rp)
    dst = np.repeat(np.arange(n), deg)
    src = np.asarray(ci, np.int64)
    P = np.empty((len(src), heads))
    logit = np.empty((len(src), heads))
    for k in range(0, len(src), chunk):
        sl = slice(k, k + chunk)
        P[sl] = np.einsum("ehd,ehd->eh", g[dst[sl]], np.abs(R[src[sl]]))
        x = L[dst[sl]] + R[src[sl]]
        logit[sl] = np.einsum("ehd,hd->eh", np.where(x > 0, x, slope * x), av)
    # the weights, a softmax over each row's edges
    alpha = np.zeros_like(logit)
    if len(src):
        starts = rp[:-1][deg > 0]
        m = np.repeat(np.maximum.reduceat(logit, starts, axis=0), deg[deg > 0], axis=0)
        ex = np.exp(logit - m)
        alpha = ex / np.repeat(np.add.reduceat(ex, starts, axis=0), deg[deg > 0], axis=0)
    def seg(idx, wts):  # sums of wts over the edges grouped by node idx
        return np.bincount(idx, weights=wts, minlength=n)

    Gabs = np.stack([seg(dst, alpha[:, h] * P[:, h]) for h in range(heads)], 1)
    wde = alpha * (P + Gabs[dst])                 # bound of |de_ij| per head
    wsum = np.stack([seg(dst, wde[:, h]) for h in range(heads)], 1)
    S_l = (wsum[:, :, None] * aa[None]).reshape(n, HD)
    S_r = np.zeros((n, heads, D))
    for h in range(heads):
        gh = alpha[:, h, None] * g[dst, h, :]
        S_r[:, h, :] = np.stack([seg(src, gh[:, d]) for d in range(D)], 1)
        S_r[:, h, :] += seg(src, wde[:, h])[:, None] * aa[h][None]
    S_a = np.zeros((heads, D))
    for k in range(0, len(src), chunk):
        sl = slice(k, k + chunk)
        S_a += np.einsum("eh,ehd->hd", wde[sl], np.abs(L[dst[sl]] + R[src[sl]]))
    return S_l, S_r.reshape(n, HD), S_a


def check_gatv2_backward(gnn, rp, ci, heads, D, bf16, shared, seed=0, slope=0.2):
    n = len(rp) - 1
    Cl, Cr, a, dO = _gatv2_inputs(n, heads, D, bf16, shared, seed)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, lse = _gatv2_forward_exact(gnn, g, Cl, Cr, a, heads, D, slope)
    gt = _transpose_graph(gnn, rp, ci)
    dl, dr, da = gnn.gnn_gatv2_attn_bwd(g, gt, _dev_feat(Cl), None if Cr is None else _dev_feat(Cr),
                                        dev(a), heads, D, out, lse, dev(dO), slope)
    rl, rr, ra = oracle.gatv2_backward(rp, ci, Cl, Cr, a, heads, D, dO, slope)
    S_l, S_r, S_a = gatv2_term_scales(rp, ci, Cl, Cr, a, heads, D, dO, slope)
    # both sides score the same (bf16 or fp32) features, so only fp32
    # arithmetic (here and in the forward's out and lse) separates them
    what = f"gatv2 backward {heads}x{D} {'bf16' if bf16 else 'fp32'}{' shared' if shared else ''}"
    # the row-wise normwise error, reported beside the term-scaled bound the
    # test enforces (the two differ where a row's terms cancel)
    from tests.tolerance import rowwise_rel_err
    rw = [float(np.max(rowwise_rel_err(x.cpu().numpy(), r)[0], initial=0.0))
          for x, r in ((dl, rl), (dr, rr))]
    print(f"GATV2_BWD_ROWWISE {what}: dl {rw[0]:.2e} dr {rw[1]:.2e}")
    assert_terms_close(dl.cpu().numpy(), rl, S_l, TOL_F32, what + " dl")
    assert_terms_close(dr.cpu().numpy(), rr, S_r, TOL_F32, what + " dr")
    assert_terms_close(da.cpu().numpy(), ra, S_a, TOL_F32, what + " da")
    return dl, dr, da


def _hub_graph(n, seed):
    """Random edges plus a destination hub (in-degree 900: its row is cut into
    pieces over four runs of 256 edges), a source hub (out-degree 600: a
    heavy row of CSR^T) and two nodes without in-edges (empty rows)."""
    rng = np.random.default_rng(seed)
    edges = [(int(rng.integers(n)), int(rng.integers(n))) for _ in range(6 * n)]
    edges += [(int(s), 7) for s in rng.choice(n, 900, replace=False)]
    edges += [(3, int(d)) for d in rng.choice(n, 600, replace=False)]
    return G.from_edges(n, [(s, d) for s, d in edges if d not in (50, 51)], self_loops=False)


@pytest.mark.parametrize("heads,D,bf16", [(1, 32, False), (2, 32, False), (4, 32, False),
                                          (4, 64, False), (4, 64, True), (8, 32, True),
                                          (2, 32, True), (1, 32, True)])
def test_gatv2_backward_hub_graph(gnn, heads, D, bf16):
    rp, ci = _hub_graph(1200, heads * D + bf16)
    dl, dr, _ = check_gatv2_backward(gnn, rp, ci, heads, D, bf16, shared=False)
    assert not dl[50:52].any(), "rows without edges have dl = 0"


@pytest.mark.parametrize("bf16", [False, True])
def test_gatv2_backward_shared_projection(gnn, bf16):
    rp, ci = _hub_graph(1200, 5)
    check_gatv2_backward(gnn, rp, ci, 4, 64, bf16, shared=True, seed=1)


def test_gatv2_backward_rmat_power_law(gnn):
    """R-MAT scale 13: rows from one edge to hundreds, many cut at runs."""
    rp, ci = synth.rmat(13, 16)
    check_gatv2_backward(gnn, rp, ci, 4, 64, True, shared=True, seed=2)


def test_gatv2_backward_deterministic(gnn):
    rp, ci = synth.rmat(12, 16)
    n = len(rp) - 1
    Cl, Cr, a, dO = _gatv2_inputs(n, 4, 64, True, True, 3)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, lse = _gatv2_forward_exact(gnn, g, Cl, Cr, a, 4, 64, 0.2)
    gt = _transpose_graph(gnn, rp, ci)
    args = (g, gt, _dev_feat(Cl), None, dev(a), 4, 64, out, lse, dev(dO))
    first = [t.cpu().numpy() for t in gnn.gnn_gatv2_attn_bwd(*args)]
    for _ in range(2):
        again = [t.cpu().numpy() for t in gnn.gnn_gatv2_attn_bwd(*args)]
        for x, y in zip(first, again):
            assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def _subgraph(rp, ci, rows):
    """The rows `rows` with their whole edge lists, every other row emptied,
    relabelled onto the nodes they touch: (rowptr, colidx, nodes) with
    nodes[new] = old."""
    rows = np.unique(rows)
    nodes = np.unique(np.concatenate([rows] + [ci[rp[r]:rp[r + 1]] for r in rows]))
    pos = np.searchsorted(nodes, rows)
    deg = np.zeros(len(nodes), np.int64)
    deg[pos] = rp[rows + 1].astype(np.int64) - rp[rows]
    srp = np.zeros(len(nodes) + 1, np.int64)
    srp[1:] = np.cumsum(deg)
    sci = np.empty(int(srp[-1]), np.int32)
    for r, k in zip(rows, pos):
        sci[srp[k]:srp[k + 1]] = np.searchsorted(nodes, ci[rp[r]:rp[r + 1]])
    return srp.astype(np.int32), sci, nodes


def test_gatv2_backward_config3_sampled(gnn):
    """R-MAT scale 20, 4 heads x 64, bf16, one projection (the GATv2
    layer's shape), on sampled rows the oracle computes exactly: dl of a
    row needs only its own edge list; dr of a node needs every row that
    lists it, each whole (its weights and G)."""
    w = synth.workload("c3_rmat20_gatv2", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n, heads, D = len(rp) - 1, 4, 64
    Cl, _, a, dO = _gatv2_inputs(n, heads, D, True, True, 4)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    out, lse = _gatv2_forward_exact(gnn, g, Cl, None, a, heads, D, 0.2)
    gt = _transpose_graph(gnn, rp, ci)
    dl, dr, _ = gnn.gnn_gatv2_attn_bwd(g, gt, _dev_feat(Cl), None, dev(a), heads, D, out, lse, dev(dO))
    dl, dr = dl.cpu().numpy(), dr.cpu().numpy()
    del out, lse
    rng = np.random.default_rng(7)
    deg = np.diff(rp)
    # dl: random rows and the five heaviest (cut into up to ~150 pieces)
    rows = np.concatenate([rng.choice(n, 60, replace=False), np.argsort(-deg)[:5]])
    srp, sci, nodes = _subgraph(rp, ci, rows)
    rl, _, _ = oracle.gatv2_backward(srp, sci, Cl[nodes], None, a, heads, D, dO[nodes])
    S_l, _, _ = gatv2_term_scales(srp, sci, Cl[nodes], None, a, heads, D, dO[nodes])
    pos = np.searchsorted(nodes, np.unique(rows))
    assert_terms_close(dl[np.unique(rows)], rl[pos], S_l[pos], TOL_F32, "c3 dl")
    # dr: random sources of modest out-degree, every row listing them whole
    rpt, cit, _ = oracle.csr_transpose(rp, ci)
    outdeg = np.diff(rpt)
    cand = np.nonzero((outdeg > 0) & (outdeg <= 40))[0]
    js = np.unique(rng.choice(cand, 12, replace=False))
    lister = np.unique(np.concatenate([cit[rpt[j]:rpt[j + 1]] for j in js]))
    srp, sci, nodes = _subgraph(rp, ci, lister)
    _, rr, _ = oracle.gatv2_backward(srp, sci, Cl[nodes], None, a, heads, D, dO[nodes])
    _, S_r, _ = gatv2_term_scales(srp, sci, Cl[nodes], None, a, heads, D, dO[nodes])
    # one projection: the gradient of C at j is dl_j + dr_j; compare dr alone
    pos = np.searchsorted(nodes, js)
    assert_terms_close(dr[js], rr[pos], S_r[pos], TOL_F32, "c3 dr")


def test_gatv2_backward_rejects_unsupported_shapes(gnn):
    rp, ci = G.random_graph(20, 0.2, 1)
    g = gnn.graph_prepare(dev(rp), dev(ci))
    gt = _transpose_graph(gnn, rp, ci)
    f = torch.zeros((20, 96), dtype=torch.float32, device="cuda")
    a = torch.zeros((3, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(gnn.GnnError) as e:  # heads * head_dim = 96
        gnn.gnn_gatv2_attn_bwd(g, gt, f, None, a, 3, 32, f, torch.zeros((20, 3), device="cuda"), f)
    assert e.value.code == gnn.GNN_ERR_UNSUPPORTED
