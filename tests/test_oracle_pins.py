"""Pins of the CPU oracle against things other than itself: dense brute force
on tiny graphs (matrix formulation, numpy), closed forms, invariants,
hand-derived golden cases (tests/golden/) and library routines.  CPU only."""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G

GOLD = os.path.join(os.path.dirname(__file__), "golden")



def _tiny_graphs():
    out = []
    for seed, (n, p, loops) in enumerate([(7, 0.3, True), (23, 0.2, True), (40, 0.1, False),
                                          (64, 0.05, True), (33, 0.5, False)]):
        out.append(G.random_graph(n, p, seed, loops))
    out.append(G.star(17))
    out.append(G.from_edges(9, [], self_loops=False))            # all rows empty
    out.append(G.from_edges(12, [(a, b) for a in range(12) for b in range(12)]))  # complete
    out.append(G.from_edges(5, [(0, 1)], self_loops=False))      # mostly empty
    return out


def _dense_weights(A, norm, values_dense=None):
    W = A.astype(np.float64) if values_dense is None else np.where(A, values_dense, 0.0)
    d_in = A.sum(axis=1).astype(np.float64)
    d_out = A.sum(axis=0).astype(np.float64)
    if norm == oracle.NORM_LEFT:
        W = W / np.where(d_in > 0, d_in, 1.0)[:, None]
    elif norm == oracle.NORM_RIGHT:
        W = W / np.where(d_out > 0, d_out, 1.0)[None, :]
    elif norm == oracle.NORM_BOTH:
        W = W / np.sqrt(np.outer(np.where(d_in > 0, d_in, 1.0), np.where(d_out > 0, d_out, 1.0)))
    return W


# ---------------------------------------------------------------- SpMM / sum / mean

@pytest.mark.parametrize("norm", [0, 1, 2, 3])
def test_spmm_equals_dense_matmul(norm):
    rng = np.random.default_rng(norm)
    for rp, ci in _tiny_graphs():
        n = len(rp) - 1
        A = G.dense_adjacency(rp, ci)
        X = rng.standard_normal((n, 6)).astype(np.float32)
        vals = rng.uniform(0.5, 2.0, len(ci)).astype(np.float32)
        vd = np.zeros((n, n))
        for i in range(n):
            vd[i, ci[rp[i]:rp[i + 1]]] = vals[rp[i]:rp[i + 1]]
        for v, vdense in ((None, None), (vals, vd)):
            ref = _dense_weights(A, norm, vdense) @ X.astype(np.float64)
            got = oracle.spmm(rp, ci, X, norm=norm, values=v)
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_sum_of_ones_is_in_degree_exactly():
    rp, ci = G.random_graph(50, 0.2, 3)
    ones = np.ones((50, 3), np.float32)
    got = oracle.segment_reduce(oracle.OP_SUM, rp, ci, ones)
    d_in, _ = oracle.degrees(rp, ci)
    assert np.array_equal(got, np.repeat(np.diff(rp)[:, None], 3, axis=1).astype(np.float64))
    assert np.array_equal(d_in, np.diff(rp))


def test_degrees_match_dense_counts():
    for rp, ci in _tiny_graphs():
        A = G.dense_adjacency(rp, ci)
        d_in, d_out = oracle.degrees(rp, ci)
        assert np.array_equal(d_in, A.sum(axis=1))
        assert np.array_equal(d_out, A.sum(axis=0))


def test_gcn_on_regular_graph_keeps_constant_features():
    # circulant k-regular digraph + self-loops: every in- and out-degree is k+1,
    # so D^-1/2 A D^-1/2 has rows summing to 1
    n, k = 30, 4
    rp, ci = G.from_edges(n, [((i + s) % n, i) for i in range(n) for s in range(1, k + 1)])
    X = np.full((n, 5), 1.75, np.float32)
    got = oracle.spmm(rp, ci, X, norm=oracle.NORM_BOTH)
    np.testing.assert_allclose(got, 1.75, rtol=1e-14)


def test_mean_of_constant_and_mean_is_sum_over_degree():
    rp, ci = G.random_graph(40, 0.15, 5)
    X = np.full((40, 4), -0.375, np.float32)
    m = oracle.segment_reduce(oracle.OP_MEAN, rp, ci, X)
    assert np.all(m == -0.375)
    Xr = np.random.default_rng(1).standard_normal((40, 4)).astype(np.float32)
    s = oracle.segment_reduce(oracle.OP_SUM, rp, ci, Xr)
    m = oracle.segment_reduce(oracle.OP_MEAN, rp, ci, Xr)
    np.testing.assert_allclose(m, s / np.diff(rp)[:, None], rtol=1e-15)


def test_empty_rows_give_zero():
    rp, ci = G.from_edges(6, [(0, 1), (2, 1)], self_loops=False)
    X = np.arange(12, dtype=np.float32).reshape(6, 2) + 1
    for op in (oracle.OP_SUM, oracle.OP_MEAN):
        y = oracle.segment_reduce(op, rp, ci, X)
        assert np.all(y[[0, 2, 3, 4, 5]] == 0)
    y, am = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
    assert np.all(y[[0, 2, 3, 4, 5]] == 0) and np.all(am[[0, 2, 3, 4, 5]] == -1)
    assert np.all(oracle.spmm(rp, ci, X)[[0, 2, 3, 4, 5]] == 0)


def test_bf16_inputs_widen_exactly():
    rp, ci = G.random_graph(20, 0.3, 9)
    bits = np.random.default_rng(2).integers(0x3c00, 0x4100, (20, 8)).astype(np.uint16)
    bits[::3] |= 0x8000
    x32 = (bits.astype(np.uint32) << 16).view(np.float32)
    for op in (oracle.OP_SUM, oracle.OP_MEAN):
        assert np.array_equal(oracle.segment_reduce(op, rp, ci, bits),
                              oracle.segment_reduce(op, rp, ci, x32))
    assert np.array_equal(oracle.spmm(rp, ci, bits), oracle.spmm(rp, ci, x32))


# ---------------------------------------------------------------- max / argmax

def test_order_key_golden():
    rows = G.read_golden(os.path.join(GOLD, "order_key.txt"))
    with open(os.path.join(GOLD, "order_key.txt")) as f:
        pairs = [l.split() for l in f if l.strip() and not l.startswith("#")]
    floats, keys = [], []
    for b, k in pairs:
        v = np.array([int(b, 16)], np.uint32).view(np.float32)[0]
        assert oracle.order_key(float(v)) == int(k, 16), (b, k)
        floats.append(float(v))
        keys.append(int(k, 16))
    # keys order the floats (with -0 < +0)
    order_f = sorted(range(len(floats)), key=lambda i: (floats[i], math.copysign(1, floats[i])))
    assert [keys[i] for i in order_f] == sorted(keys)
    assert rows  # file parsed


def test_max_argmax_bruteforce_with_ties():
    rng = np.random.default_rng(11)
    for rp, ci in _tiny_graphs():
        n = len(rp) - 1
        A = G.dense_adjacency(rp, ci)
        X = rng.integers(-3, 4, (n, 5)).astype(np.float32)   # many ties
        y, am = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
        for i in range(n):
            nb = np.nonzero(A[i])[0]          # ascending ids
            for f in range(5):
                if len(nb) == 0:
                    assert y[i, f] == 0 and am[i, f] == -1
                    continue
                vals = X[nb, f]
                best = vals.max()
                assert y[i, f] == best
                assert am[i, f] == nb[np.nonzero(vals == best)[0][0]]   # smallest id


def test_max_orders_negative_zero_below_positive_zero():
    rp, ci = G.from_edges(3, [(0, 2), (1, 2)], self_loops=False)
    X = np.array([[-0.0], [0.0], [5.0]], np.float32)
    y, am = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
    assert am[2, 0] == 1 and y[2, 0] == 0.0 and math.copysign(1, y[2, 0]) == 1.0
    X = np.array([[0.0], [-0.0], [5.0]], np.float32)
    y, am = oracle.segment_reduce(oracle.OP_MAX, rp, ci, X)
    assert am[2, 0] == 0


def test_min_argmin_bruteforce_with_ties_and_signed_zero():
    """min by plain comparison (value, then -0 before +0, then smallest id),
    written without the order key."""
    rng = np.random.default_rng(12)
    for rp, ci in _tiny_graphs():
        n = len(rp) - 1
        A = G.dense_adjacency(rp, ci)
        X = rng.integers(-3, 4, (n, 5)).astype(np.float32)
        X[rng.random(X.shape) < 0.25] = -0.0
        y, am = oracle.segment_reduce(oracle.OP_MIN, rp, ci, X)
        for i in range(n):
            nb = np.nonzero(A[i])[0]
            for f in range(5):
                if len(nb) == 0:
                    assert y[i, f] == 0 and am[i, f] == -1
                    continue
                best = min(nb, key=lambda j: (float(X[j, f]), 0 if math.copysign(1, X[j, f]) < 0 else 1, j))
                assert am[i, f] == best
                assert y[i, f] == X[best, f] and math.copysign(1, y[i, f]) == math.copysign(1, X[best, f])


def test_min_is_negated_max_of_negation():
    """min(X) = -max(-X), argmin = argmax of -X: negation reverses the order
    of every pair of values (-0 and +0 included) and keeps the ids."""
    rng = np.random.default_rng(13)
    rp, ci = G.random_graph(60, 0.1, 5)
    X = rng.integers(-4, 5, (60, 6)).astype(np.float32)
    X[rng.random(X.shape) < 0.2] = -0.0
    y, am = oracle.segment_reduce(oracle.OP_MIN, rp, ci, X)
    y2, am2 = oracle.segment_reduce(oracle.OP_MAX, rp, ci, -X)
    empty = np.diff(rp) == 0
    assert np.array_equal(am, am2)
    assert np.array_equal(np.signbit(y[~empty]), np.signbit(-y2[~empty])) and np.array_equal(y, -y2)


@pytest.mark.parametrize("op", ["max", "min"])
def test_reduce_backward_matches_finite_differences(op):
    """d/dX of sum(g * reduce(X)) by finite differences of the forward
    oracle, on a tie-free input (values 0.1 apart, step 2^-10)."""
    rng = np.random.default_rng(31)
    rp, ci = G.random_graph(12, 0.35, 6)
    n, F = 12, 3
    X = (rng.permutation(n * F).reshape(n, F) * 0.1).astype(np.float32)
    g = rng.standard_normal((n, F))
    code = oracle.OP_MAX if op == "max" else oracle.OP_MIN
    y, arg = oracle.segment_reduce(code, rp, ci, X)
    gx = oracle.reduce_ext_backward(arg, g, n)
    eps = 2.0 ** -10
    base = float(np.sum(g * y))
    num = np.zeros((n, F))
    for j in range(n):
        for f in range(F):
            Xp = X.copy()
            Xp[j, f] += eps
            yp, _ = oracle.segment_reduce(code, rp, ci, Xp)
            num[j, f] = (float(np.sum(g * yp)) - base) / eps
    assert np.allclose(gx, num, rtol=1e-6, atol=1e-6)


def test_reduce_backward_empty_rows_and_shared_sources():
    # arg -1 rows contribute nothing; a source that is the max of several
    # rows collects all their gradients
    arg = np.array([[2, -1], [2, 0], [-1, 0]], np.int32)
    go = np.array([[1.0, 5.0], [2.0, 3.0], [7.0, 4.0]])
    gx = oracle.reduce_ext_backward(arg, go, 3)
    assert np.array_equal(gx, [[0.0, 7.0], [0.0, 0.0], [3.0, 0.0]])


def test_csr_transpose_is_the_transposed_adjacency_and_an_involution():
    for rp, ci in _tiny_graphs():
        n = len(rp) - 1
        rpt, cit, _ = oracle.csr_transpose(rp, ci)
        assert np.array_equal(G.dense_adjacency(rpt, cit), G.dense_adjacency(rp, ci).T)
        rp2, ci2, _ = oracle.csr_transpose(rpt, cit)
        assert np.array_equal(rp2, rp) and np.array_equal(ci2, ci)
    # rectangular, with values following their edges
    rp = np.array([0, 2, 3], np.int32)
    ci = np.array([1, 4, 0], np.int32)
    vals = np.array([0.5, 2.0, 3.0], np.float32)
    rpt, cit, vt = oracle.csr_transpose(rp, ci, n_cols=5, values=vals)
    assert np.array_equal(rpt, [0, 1, 2, 2, 2, 3]) and np.array_equal(cit, [1, 0, 0])
    assert np.array_equal(vt, [3.0, 0.5, 2.0])


@pytest.mark.parametrize("norm,spmm_norm", [(oracle.NORM_BOTH, oracle.NORM_BOTH),
                                            (oracle.NORM_NONE, oracle.NORM_NONE),
                                            (oracle.NORM_LEFT, oracle.NORM_RIGHT)])
def test_spmm_backward_is_spmm_on_the_transpose(norm, spmm_norm):
    """d/dX of sum(G * spmm(A, X)) = (normalised A)^T G, built densely, equals
    the SpMM on CSR^T: GCN with BOTH, sum with NONE, mean (LEFT) with RIGHT."""
    rng = np.random.default_rng(41)
    rp, ci = G.random_graph(30, 0.15, 8)
    n = 30
    A = G.dense_adjacency(rp, ci).astype(np.float64)
    din, dout = A.sum(1), A.sum(0)
    with np.errstate(divide="ignore"):
        if norm == oracle.NORM_BOTH:
            An = A * np.where(din > 0, din ** -0.5, 0)[:, None] * np.where(dout > 0, dout ** -0.5, 0)[None, :]
        elif norm == oracle.NORM_LEFT:
            An = A * np.where(din > 0, 1.0 / din, 0)[:, None]
        else:
            An = A
    Gy = rng.standard_normal((n, 4))
    rpt, cit, _ = oracle.csr_transpose(rp, ci)
    got = oracle.spmm(rpt, cit, Gy.astype(np.float32), norm=spmm_norm)
    assert np.allclose(got, An.T @ Gy.astype(np.float32).astype(np.float64), rtol=1e-12, atol=1e-12)


def test_gt_backward_matches_finite_differences():
    """dQ, dK, dV of sum(dO * GT(Q, K, V)) by central differences of the
    forward oracle on a small graph (2 heads x 4)."""
    rng = np.random.default_rng(51)
    rp, ci = G.random_graph(9, 0.4, 9)
    n, heads, D, scale = 9, 2, 4, 0.7
    # fp32 inputs (the oracle's input type) and a step they represent exactly
    Q, K, V = (rng.standard_normal((n, heads * D)).astype(np.float32) for _ in range(3))
    dO = rng.standard_normal((n, heads * D))
    dQ, dK, dV = oracle.gt_backward(rp, ci, Q, K, V, heads, D, scale, dO)

    def loss(Qx, Kx, Vx):
        out, _ = oracle.gt(rp, ci, Qx, Kx, Vx, heads, D, scale)
        return float(np.sum(dO * out))

    eps = 2.0 ** -10
    for got, which in ((dQ, 0), (dK, 1), (dV, 2)):
        num = np.zeros_like(got)
        for idx in np.ndindex(*got.shape):
            args_p = [Q.copy(), K.copy(), V.copy()]
            args_m = [Q.copy(), K.copy(), V.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert np.allclose(got, num, rtol=1e-4, atol=1e-6), ("dQ", "dK", "dV")[which]
    # every row's weights sum to 1, so dV summed over the sources is dO summed
    # over the rows with edges
    has = np.diff(rp) > 0
    assert np.allclose(dV.sum(0), dO[has].sum(0), rtol=1e-12, atol=1e-12)


def _gatv2_grid_features(rng, n, HD):
    """l and r on the grid k/8 + 1/32: every l_i + r_j sits at least 1/16
    from LeakyReLU's kink, so a step of 2^-10 never crosses it."""
    return tuple((rng.integers(-12, 13, (n, HD)) / 8 + 1 / 32).astype(np.float32)
                 for _ in range(2))


def test_gatv2_backward_matches_finite_differences():
    """dl, dr, da of sum(dO * GATv2(l, r)) by central differences of the
    forward oracle (2 heads x 4, separate left and right projections):
    H = [l | r] with W_l = [I; 0], W_r = [0; I] makes the projected rows l
    and r themselves."""
    rng = np.random.default_rng(53)
    rp, ci = G.random_graph(9, 0.4, 11)
    n, heads, D, slope = 9, 2, 4, 0.2
    HD = heads * D
    l, r = _gatv2_grid_features(rng, n, HD)
    a = rng.standard_normal((heads, D)).astype(np.float32)
    dO = rng.standard_normal((n, HD))
    dl, dr, da = oracle.gatv2_backward(rp, ci, l, r, a, heads, D, dO, slope)
    eye, zero = np.eye(HD, dtype=np.float32), np.zeros((HD, HD), np.float32)
    W_l, W_r = np.vstack([eye, zero]), np.vstack([zero, eye])

    def loss(lx, rx, ax):
        out, _ = oracle.gatv2(rp, ci, np.hstack([lx, rx]), W_l, ax, heads, D, slope, W_r=W_r)
        return float(np.sum(dO * out))

    eps = 2.0 ** -10
    for got, which in ((dl, 0), (dr, 1), (da, 2)):
        num = np.zeros_like(got)
        for idx in np.ndindex(*got.shape):
            args_p = [l.copy(), r.copy(), a.copy()]
            args_m = [l.copy(), r.copy(), a.copy()]
            args_p[which][idx] += eps
            args_m[which][idx] -= eps
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        assert np.allclose(got, num, rtol=1e-4, atol=1e-6), ("dl", "dr", "da")[which]


def test_gatv2_backward_shared_projection_is_dl_plus_dr():
    """With one projection (r = l = C) the gradient of C is dl + dr: central
    differences of the forward with H = C, W = I (1 head x 8, a hub row)."""
    rng = np.random.default_rng(54)
    n, heads, D, slope = 8, 1, 8, 0.2
    rp, ci = G.from_edges(n, [(s, 0) for s in range(1, n)] + [(2, 5), (6, 3), (4, 7)])
    C, _ = _gatv2_grid_features(rng, n, D)
    a = rng.standard_normal((heads, D)).astype(np.float32)
    dO = rng.standard_normal((n, D))
    dl, dr, _ = oracle.gatv2_backward(rp, ci, C, None, a, heads, D, dO, slope)
    eye = np.eye(D, dtype=np.float32)
    eps = 2.0 ** -10
    num = np.zeros((n, D))
    for idx in np.ndindex(n, D):
        cp, cm = C.copy(), C.copy()
        cp[idx] += eps
        cm[idx] -= eps
        num[idx] = (np.sum(dO * oracle.gatv2(rp, ci, cp, eye, a, heads, D, slope)[0]) -
                    np.sum(dO * oracle.gatv2(rp, ci, cm, eye, a, heads, D, slope)[0])) / (2 * eps)
    assert np.allclose(dl + dr, num, rtol=1e-4, atol=1e-6)


def test_gatv2_backward_special_cases():
    """slope 1: LeakyReLU is the identity, the logit's l_i part is constant
    over the row and cancels in the softmax, so dl = 0.  a = 0: uniform
    weights, dl = 0, da is still defined and dr_j = sum over the rows i that
    list j of dO_i / deg(i)."""
    rng = np.random.default_rng(55)
    rp, ci = G.random_graph(30, 0.2, 12)
    n, heads, D = 30, 2, 4
    HD = heads * D
    l, r = (rng.standard_normal((n, HD)).astype(np.float32) for _ in range(2))
    a = rng.standard_normal((heads, D)).astype(np.float32)
    dO = rng.standard_normal((n, HD))
    dl, _, _ = oracle.gatv2_backward(rp, ci, l, r, a, heads, D, dO, 1.0)
    assert np.max(np.abs(dl)) < 1e-12
    dl0, dr0, _ = oracle.gatv2_backward(rp, ci, l, r, np.zeros_like(a), heads, D, dO, 0.2)
    assert np.max(np.abs(dl0)) == 0.0
    want = np.zeros((n, HD))
    for i in range(n):
        deg = rp[i + 1] - rp[i]
        for j in ci[rp[i]:rp[i + 1]]:
            want[j] += dO[i] / deg
    assert np.allclose(dr0, want, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- degree statistics

def _rowptr_of(deg):
    rp = np.zeros(len(deg) + 1, np.int32)
    rp[1:] = np.cumsum(deg)
    return rp


def test_degree_stats_regular_graph():
    """Every row of length 7: mean 7, no spread, skewness 0 by convention."""
    assert oracle.degree_stats(_rowptr_of([7] * 50)) == (7.0, 0.0, 0.0, 7.0)


def test_degree_stats_two_point_closed_form():
    """One row of length k, n - 1 rows of length 1: a two-point law with
    p = 1/n, whose skewness is (1 - 2p) / sqrt(p (1 - p)) and standard
    deviation (k - 1) sqrt(p (1 - p))."""
    n, k = 40, 301
    mean, std, skew, mx = oracle.degree_stats(_rowptr_of([k] + [1] * (n - 1)))
    p = 1.0 / n
    assert mx == k
    assert mean == pytest.approx(1 + (k - 1) * p, rel=1e-15)
    assert std == pytest.approx((k - 1) * np.sqrt(p * (1 - p)), rel=1e-13)
    assert skew == pytest.approx((1 - 2 * p) / np.sqrt(p * (1 - p)), rel=1e-13)


def test_degree_stats_matches_scipy():
    """Power-law row lengths (R-MAT scale 12): scipy's biased sample
    skewness and numpy's population deviation."""
    stats = pytest.importorskip("scipy.stats")
    rp, _ = synth.rmat(12, 16)
    d = np.diff(rp).astype(np.float64)
    mean, std, skew, mx = oracle.degree_stats(rp)
    assert mean == pytest.approx(d.mean(), rel=1e-14)
    assert std == pytest.approx(d.std(), rel=1e-12)
    assert skew == pytest.approx(stats.skew(d, bias=True), rel=1e-10)
    assert mx == d.max()


def test_backward_and_statistics_degenerate_graphs():
    """No edges: every gradient is zero (no weight, no score).  A single
    self-loop row: its weight is 1, so the score gradient vanishes and dr of
    the node is dO.  No nodes: statistics are zero."""
    rng = np.random.default_rng(56)
    n, heads, D = 6, 2, 4
    HD = heads * D
    rp, ci = G.from_edges(n, [], self_loops=False)
    l, r = (rng.standard_normal((n, HD)).astype(np.float32) for _ in range(2))
    a = rng.standard_normal((heads, D)).astype(np.float32)
    dO = rng.standard_normal((n, HD))
    for out in oracle.gatv2_backward(rp, ci, l, r, a, heads, D, dO):
        assert not np.any(out)
    for out in oracle.gt_backward(rp, ci, l, r, r, heads, D, 0.5, dO):
        assert not np.any(out)
    rp1, ci1 = G.from_edges(n, [], self_loops=True)
    dl, dr, da = oracle.gatv2_backward(rp1, ci1, l, r, a, heads, D, dO)
    assert not np.any(dl) and not np.any(da) and np.array_equal(dr, dO)
    assert oracle.degree_stats(np.zeros(1, np.int32)) == (0.0, 0.0, 0.0, 0.0)


# ---------------------------------------------------------------- relabel invariance

@pytest.mark.parametrize("op", ["spmm", "sum", "mean", "max"])
def test_relabel_invariance(op):
    rng = np.random.default_rng(21)
    rp, ci = G.random_graph(45, 0.12, 4)
    n = 45
    X = rng.integers(-2, 3, (n, 4)).astype(np.float32) if op == "max" else \
        rng.standard_normal((n, 4)).astype(np.float32)
    p = rng.permutation(n).astype(np.int32)
    rp2, ci2 = G.relabel(rp, ci, p)
    X2 = X[p]

    def run(r, c, x):
        if op == "spmm":
            return oracle.spmm(r, c, x, norm=oracle.NORM_BOTH), None
        if op == "max":
            return oracle.segment_reduce(oracle.OP_MAX, r, c, x)
        return oracle.segment_reduce(oracle.OP_SUM if op == "sum" else oracle.OP_MEAN, r, c, x), None

    y, am = run(rp, ci, X)
    y2, am2 = run(rp2, ci2, X2)
    np.testing.assert_allclose(y2, y[p], rtol=1e-12, atol=1e-14)
    if op == "max":
        # argmax: same value at the mapped source; ties re-resolved under new ids
        inv = np.empty(n, np.int64)
        inv[p] = np.arange(n)
        A2 = G.dense_adjacency(rp2, ci2)
        for r in range(n):
            for f in range(4):
                nb = np.nonzero(A2[r])[0]
                best = X2[nb, f].max()
                assert am2[r, f] == nb[np.nonzero(X2[nb, f] == best)[0][0]]
                assert X[p[am2[r, f]], f] == X[am[p[r], f], f]


# ---------------------------------------------------------------- GATv2

def _dense_gatv2(A, C_l, C_r, a, heads, D, slope):
    n = A.shape[0]
    out = np.zeros((n, heads * D))
    lse = np.full((n, heads), -np.inf)
    alpha = np.zeros((n, n, heads))
    for h in range(heads):
        s = slice(h * D, (h + 1) * D)
        X = C_l[:, None, s] + C_r[None, :, s]           # [i, j, d]
        E = (np.where(X > 0, X, slope * X) * a[h][None, None, :]).sum(-1)
        E = np.where(A, E, -np.inf)
        m = E.max(axis=1, keepdims=True)
        ok = np.isfinite(m[:, 0])
        P = np.where(A, np.exp(E - np.where(np.isfinite(m), m, 0)), 0.0)
        Z = P.sum(axis=1, keepdims=True)
        al = np.where(ok[:, None], P / np.where(Z > 0, Z, 1), 0)
        alpha[:, :, h] = al
        out[:, s] = al @ C_r[:, s]
        lse[ok, h] = (m[:, 0] + np.log(Z[:, 0]))[ok]
    return out, lse, alpha


@pytest.mark.parametrize("heads,D,shared", [(1, 4, True), (2, 3, False), (3, 2, True)])
def test_gatv2_dense_bruteforce(heads, D, shared):
    rng = np.random.default_rng(heads * 10 + D)
    for rp, ci in _tiny_graphs()[:6]:
        n = len(rp) - 1
        if np.any(np.diff(rp) == 0):
            continue
        A = G.dense_adjacency(rp, ci)
        F = 5
        H = rng.standard_normal((n, F)).astype(np.float32)
        Wl = rng.standard_normal((F, heads * D)).astype(np.float32)
        Wr = Wl if shared else rng.standard_normal((F, heads * D)).astype(np.float32)
        a = rng.standard_normal((heads, D)).astype(np.float32)
        out, lse, alpha = oracle.gatv2(rp, ci, H, Wl, a, heads, D, 0.2,
                                       W_r=None if shared else Wr, want_alpha=True)
        H64 = H.astype(np.float64)
        ro, rl, ra = _dense_gatv2(A, H64 @ Wl.astype(np.float64), H64 @ Wr.astype(np.float64),
                                  a.astype(np.float64), heads, D, 0.2)
        np.testing.assert_allclose(out, ro, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)
        # alpha rows sum to one; CSR-order alpha equals the dense one
        pos = 0
        for i in range(n):
            nb = ci[rp[i]:rp[i + 1]]
            np.testing.assert_allclose(alpha[pos:pos + len(nb)], ra[i, nb], rtol=1e-10, atol=1e-14)
            np.testing.assert_allclose(alpha[pos:pos + len(nb)].sum(0), 1.0, rtol=1e-12)
            pos += len(nb)


def test_gatv2_golden_two_nodes():
    g = G.read_golden(os.path.join(GOLD, "gatv2_2node.txt"))
    f = lambda k: np.array([float(x) for x in g[k]])
    rp = f("rowptr").astype(np.int32)
    ci = f("colidx").astype(np.int32)
    out, lse = oracle.gatv2(rp, ci, f("H").reshape(2, 2).astype(np.float32),
                            f("W").reshape(2, 2).astype(np.float32), f("a").reshape(1, 2), 1, 2, 0.2)
    np.testing.assert_allclose(out[0], f("out0"), atol=1e-14)
    np.testing.assert_allclose(out[1], f("out1"), atol=1e-14)
    np.testing.assert_allclose(lse[:, 0], [f("lse0")[0], f("lse1")[0]], atol=1e-14)


def test_gatv2_zero_attention_vector_gives_neighbour_mean():
    # a = 0 -> uniform alpha -> out = mean of r over N(i); integer H and W keep
    # C = H W exact in fp32 so the mean can come from the segment-mean oracle
    rng = np.random.default_rng(3)
    rp, ci = G.random_graph(30, 0.2, 8)
    H = rng.integers(-3, 4, (30, 4)).astype(np.float32)
    W = rng.integers(-2, 3, (4, 6)).astype(np.float32)
    out, _ = oracle.gatv2(rp, ci, H, W, np.zeros((2, 3), np.float32), 2, 3, 0.2)
    C = (H.astype(np.float64) @ W.astype(np.float64)).astype(np.float32)
    ref = oracle.segment_reduce(oracle.OP_MEAN, rp, ci, C)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_gatv2_self_loop_only_row_returns_own_projection():
    rp, ci = G.from_edges(4, [(0, 1), (2, 1)])   # rows 0, 2, 3 have only their self-loop
    rng = np.random.default_rng(4)
    H = rng.standard_normal((4, 3)).astype(np.float32)
    W = rng.standard_normal((3, 4)).astype(np.float32)
    out, _ = oracle.gatv2(rp, ci, H, W, rng.standard_normal((2, 2)).astype(np.float32), 2, 2, 0.2)
    C = H.astype(np.float64) @ W.astype(np.float64)
    np.testing.assert_allclose(out[[0, 2, 3]], C[[0, 2, 3]], rtol=1e-13)


def test_gatv2_slope_one_makes_alpha_independent_of_left_projection():
    rng = np.random.default_rng(6)
    rp, ci = G.random_graph(25, 0.25, 2)
    H = rng.standard_normal((25, 4)).astype(np.float32)
    Wr = rng.standard_normal((4, 6)).astype(np.float32)
    a = rng.standard_normal((2, 3)).astype(np.float32)
    _, _, al1 = oracle.gatv2(rp, ci, H, rng.standard_normal((4, 6)).astype(np.float32), a, 2, 3,
                             1.0, W_r=Wr, want_alpha=True)
    _, _, al2 = oracle.gatv2(rp, ci, H, rng.standard_normal((4, 6)).astype(np.float32), a, 2, 3,
                             1.0, W_r=Wr, want_alpha=True)
    np.testing.assert_allclose(al1, al2, rtol=1e-11, atol=1e-14)


# ---------------------------------------------------------------- Graph Transformer

def test_gt_dense_bruteforce():
    rng = np.random.default_rng(12)
    heads, D, s = 2, 4, 0.5
    for rp, ci in _tiny_graphs()[:6]:
        n = len(rp) - 1
        if np.any(np.diff(rp) == 0):
            continue
        A = G.dense_adjacency(rp, ci)
        Q, K, V = (rng.standard_normal((n, heads * D)).astype(np.float32) for _ in range(3))
        out, lse, alpha = oracle.gt(rp, ci, Q, K, V, heads, D, s, want_alpha=True)
        for h in range(heads):
            sl = slice(h * D, (h + 1) * D)
            E = s * (Q[:, sl].astype(np.float64) @ K[:, sl].astype(np.float64).T)
            E = np.where(A, E, -np.inf)
            m = E.max(1, keepdims=True)
            P = np.where(A, np.exp(E - m), 0)
            Z = P.sum(1, keepdims=True)
            np.testing.assert_allclose(out[:, sl], (P / Z) @ V[:, sl].astype(np.float64),
                                       rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(lse[:, h], np.log(np.exp(E).sum(1)), rtol=1e-12)
        pos = 0
        for i in range(n):
            d = rp[i + 1] - rp[i]
            np.testing.assert_allclose(alpha[pos:pos + d].sum(0), 1.0, rtol=1e-12)
            pos += d


def test_gt_golden_two_nodes():
    g = G.read_golden(os.path.join(GOLD, "gt_2node.txt"))
    f = lambda k: np.array([float(x) for x in g[k]])
    rp = f("rowptr").astype(np.int32)
    ci = f("colidx").astype(np.int32)
    Q, K, V = (f(k).reshape(2, 2).astype(np.float32) for k in "QKV")
    out, lse = oracle.gt(rp, ci, Q, K, V, 1, 2, f("scale")[0])
    np.testing.assert_allclose(out[0], f("out0"), atol=1e-14)
    np.testing.assert_allclose(out[1], f("out1"), atol=1e-14)
    np.testing.assert_allclose(lse[:, 0], [f("lse0")[0], f("lse1")[0]], atol=1e-14)


def test_gt_zero_query_is_mean_of_values_and_equal_keys_uniform():
    rng = np.random.default_rng(13)
    rp, ci = G.random_graph(30, 0.2, 6)
    V = rng.standard_normal((30, 6)).astype(np.float32)
    K = rng.standard_normal((30, 6)).astype(np.float32)
    out, _ = oracle.gt(rp, ci, np.zeros((30, 6), np.float32), K, V, 2, 3, 0.7)
    ref = oracle.segment_reduce(oracle.OP_MEAN, rp, ci, V)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    Kc = np.tile(rng.standard_normal((1, 6)).astype(np.float32), (30, 1))
    _, _, al = oracle.gt(rp, ci, rng.standard_normal((30, 6)).astype(np.float32), Kc, V, 2, 3,
                         0.7, want_alpha=True)
    deg = np.repeat(np.diff(rp), np.diff(rp))
    np.testing.assert_allclose(al, np.repeat((1.0 / deg)[:, None], 2, axis=1), rtol=1e-12)


# ---------------------------------------------------------------- block-sparse tiles

def _dense_blocksparse(rp, ci, thr, packing=0):
    """Independent dense formulation of the tile decomposition (packing 1:
    columns by descending edge count in the group, ties by id)."""
    n = len(rp) - 1
    A = G.dense_adjacency(rp, ci)
    groups = []
    for g in range((n + 127) // 128):
        r0, r1 = 128 * g, min(128 * g + 128, n)
        U = np.nonzero(A[r0:r1].any(axis=0))[0]
        if packing == 1:
            cnt = A[r0:r1].sum(axis=0)[U]
            U = U[np.lexsort((U, -cnt))]
        blocks = []
        for b in range((len(U) + 15) // 16):
            cols = U[16 * b:16 * b + 16]
            tiles = []
            for w in range(8):
                sub = np.zeros((16, 16), bool)
                rr = np.arange(r0 + 16 * w, min(r0 + 16 * w + 16, r1))
                if len(rr):
                    sub[:len(rr), :len(cols)] = A[np.ix_(rr, cols)]
                p = int(sub.sum())
                kept = p >= 1 and np.float32(p) / np.float32(256) >= np.float32(thr)
                tiles.append((sub, kept))
            blocks.append((cols, tiles))
        groups.append(blocks)
    return A, groups


@pytest.mark.parametrize("packing", [oracle.PACK_ID, oracle.PACK_COUNT])
@pytest.mark.parametrize("thr", [0.0, 0.02, 0.05, 0.5, 1.0])
def test_blocksparse_matches_dense_enumeration(thr, packing):
    rng = np.random.default_rng(1)
    cases = [G.random_graph(300, 0.03, 5), G.star(150), G.from_edges(40, [], True),
             G.from_edges(130, [((i * 7) % 130, i) for i in range(130)] +
                          [(j, i) for i in range(16) for j in range(16)]),
             synth.clustered(2, 128, 0.3, 0.05, 2)]
    for rp, ci in cases:
        bs = oracle.blocksparse(rp, ci, thr, packing)
        A, groups = _dense_blocksparse(rp, ci, thr, packing)
        n = len(rp) - 1
        covered = np.zeros_like(A)
        k = 0
        for g, blocks in enumerate(groups):
            assert bs["grp_blk_offset"][g] == k
            for cols, tiles in blocks:
                if not any(kept for _, kept in tiles):
                    continue
                exp_cols = np.zeros(16, np.int32)
                exp_cols[:len(cols)] = cols
                assert np.array_equal(bs["blk_cols"][k], exp_cols)
                for w, (sub, kept) in enumerate(tiles):
                    words = bs["blk_mask"][k, w]
                    bits = np.array([(int(words[q // 64]) >> (q % 64)) & 1 for q in range(256)],
                                    bool).reshape(16, 16)
                    assert np.array_equal(bits, sub if kept else np.zeros_like(sub))
                    if kept:
                        rr = np.arange(128 * g + 16 * w, min(128 * g + 16 * w + 16, n))
                        covered[np.ix_(rr, cols)] |= sub[:len(rr), :len(cols)]
                k += 1
        assert bs["grp_blk_offset"][-1] == k == bs["n_blocks"]
        res = G.dense_adjacency(bs["res_rowptr"], bs["res_colidx"])
        # every edge exactly once across kept tiles and the residual
        assert not np.any(covered & res)
        assert np.array_equal(covered | res, A)
        assert int(covered.sum()) == bs["nnz_tiles"]
        assert bs["nnz_tiles"] + bs["nnz_residual"] == len(ci)
        for i in range(n):   # residual columns ascending
            seg = bs["res_colidx"][bs["res_rowptr"][i]:bs["res_rowptr"][i + 1]]
            assert np.all(np.diff(seg) > 0)


def test_count_packing_keeps_the_blocks_and_fills_tiles():
    """Count packing moves the same columns: at threshold 0 the listed blocks
    and tile edges equal those of id packing; along each group's packed
    order the edge counts never rise; and on a clustered graph (p = 0.3)
    more tiles reach 40% fill than with id packing."""
    rp, ci = synth.clustered(8, 256, 0.3, 0.01, 4)
    A = G.dense_adjacency(rp, ci)
    by_id = oracle.blocksparse(rp, ci, 0.0, oracle.PACK_ID)
    by_cnt = oracle.blocksparse(rp, ci, 0.0, oracle.PACK_COUNT)
    assert by_cnt["n_blocks"] == by_id["n_blocks"] and by_cnt["nnz_tiles"] == len(ci)
    off = by_cnt["grp_blk_offset"]
    n = len(rp) - 1
    for g in range(len(off) - 1):
        r0, r1 = 128 * g, min(128 * g + 128, n)
        cnt = A[r0:r1].sum(axis=0)
        cols = by_cnt["blk_cols"][off[g]:off[g + 1]].reshape(-1)
        real = cols[:int(np.count_nonzero(cnt))]
        assert np.all(np.diff(cnt[real]) <= 0)
    kept_id = oracle.blocksparse(rp, ci, 0.4, oracle.PACK_ID)["n_tiles_kept"]
    kept_cnt = oracle.blocksparse(rp, ci, 0.4, oracle.PACK_COUNT)["n_tiles_kept"]
    assert kept_cnt > 10 * max(kept_id, 1)


# ---------------------------------------------------------------- orderings

def _bandwidth(rp, ci):
    return max((abs(int(i) - int(j)) for i in range(len(rp) - 1)
                for j in ci[rp[i]:rp[i + 1]]), default=0)


def test_splitmix64_three_implementations_agree():
    import synth

    def ref(x):  # the published SplitMix64 step, written from its definition
        z = (x + 0x9E3779B97F4A7C15) & (2 ** 64 - 1)
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2 ** 64 - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2 ** 64 - 1)
        return z ^ (z >> 31)

    for x in [0, 1, 7, 2 ** 63, 2 ** 64 - 1, 0x123456789ABCDEF]:
        assert oracle.splitmix64(x) == synth.splitmix64(x) == ref(x)


def test_random_order_is_sorted_by_hash_then_id():
    rp, ci = G.random_graph(200, 0.02, 3)
    p = oracle.perm(oracle.PERM_RANDOM, rp, ci, seed=7)
    assert sorted(p.tolist()) == list(range(200))
    keys = [(oracle.splitmix64(7 ^ int(i)), int(i)) for i in p]
    assert keys == sorted(keys)


def test_degree_order_monotone_and_golden():
    rp, ci = G.random_graph(120, 0.04, 9)
    p = oracle.perm(oracle.PERM_DEGREE, rp, ci)
    A = G.dense_adjacency(rp, ci)
    deg = A.sum(0) + A.sum(1)
    assert sorted(p.tolist()) == list(range(120))
    assert all((deg[p[k]] > deg[p[k + 1]]) or (deg[p[k]] == deg[p[k + 1]] and p[k] < p[k + 1])
               for k in range(119))
    g = G.read_golden(os.path.join(GOLD, "rcm_8node.txt"))
    rp8 = np.array(g["rowptr"], np.int32)
    ci8 = np.array(g["colidx"], np.int32)
    assert oracle.perm(oracle.PERM_DEGREE, rp8, ci8).tolist() == [int(x) for x in g["degree"]]


def test_rcm_golden_eight_nodes():
    g = G.read_golden(os.path.join(GOLD, "rcm_8node.txt"))
    rp = np.array(g["rowptr"], np.int32)
    ci = np.array(g["colidx"], np.int32)
    assert oracle.perm(oracle.PERM_RCM, rp, ci).tolist() == [int(x) for x in g["rcm"]]


def test_rcm_recovers_path_and_grid_bandwidth():
    rng = np.random.default_rng(5)
    rp, ci = G.path(60)
    s = rng.permutation(60)
    rp2, ci2 = G.relabel(rp, ci, s)
    assert _bandwidth(rp2, ci2) > 1
    p = oracle.perm(oracle.PERM_RCM, rp2, ci2)
    rp3, ci3 = oracle.apply_perm(rp2, ci2, p)
    assert _bandwidth(rp3, ci3) == 1
    w = 9
    rp, ci = G.grid(w)
    s = rng.permutation(w * w)
    rp2, ci2 = G.relabel(rp, ci, s)
    p = oracle.perm(oracle.PERM_RCM, rp2, ci2)
    rp3, ci3 = oracle.apply_perm(rp2, ci2, p)
    assert _bandwidth(rp3, ci3) <= w


def _component_starts(order, S):
    """Nodes of a breadth-first order with no neighbour earlier in it."""
    pos = np.empty(len(order), np.int64)
    pos[order] = np.arange(len(order))
    return [int(u) for u in order if not np.any(S[u] & (pos < pos[u]))]


def test_rcm_matches_scipy_where_component_starts_agree():
    # scipy's reverse_cuthill_mckee also expands each BFS level by ascending
    # degree; it picks among equal-degree start nodes in its own order, so
    # the sequences are compared wherever both started the same components
    sp = pytest.importorskip("scipy.sparse")
    csgraph = pytest.importorskip("scipy.sparse.csgraph")
    checked = 0
    for seed in range(30):
        rp, ci = G.random_graph(80, 0.03, 100 + seed)
        A = G.dense_adjacency(rp, ci)
        S = (A | A.T) & ~np.eye(80, dtype=bool)
        ours = oracle.perm(oracle.PERM_RCM, rp, ci)
        theirs = csgraph.reverse_cuthill_mckee(sp.csr_matrix(S.astype(np.int8)),
                                               symmetric_mode=True)
        assert sorted(ours.tolist()) == list(range(80))
        if _component_starts(ours[::-1], S) == _component_starts(theirs[::-1], S):
            assert np.array_equal(ours, theirs)
            checked += 1
    assert checked >= 20


def test_apply_perm_matches_plain_relabel_and_commutes_with_spmm():
    rng = np.random.default_rng(17)
    rp, ci = G.random_graph(70, 0.08, 12)
    p = rng.permutation(70).astype(np.int32)
    rpo, cio = oracle.apply_perm(rp, ci, p)
    rpr, cir = G.relabel(rp, ci, p)
    assert np.array_equal(rpo, rpr) and np.array_equal(cio, cir)
    X = rng.standard_normal((70, 3)).astype(np.float32)
    np.testing.assert_allclose(oracle.spmm(rpo, cio, X[p]), oracle.spmm(rp, ci, X)[p], rtol=1e-12,
                               atol=1e-14)


def _bf16_rne_of_f32(x64):
    """fp64 -> nearest fp32 -> nearest bf16 (ties to even), as bit patterns."""
    u = np.asarray(x64, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return (u >> 16).astype(np.uint16)


def test_gatv2_rounded_projection_mode_equals_exact_mode_on_rounded_features():
    """The diagnostic mode (projected features rounded to bf16 before the
    attention, as the bf16 path stores them) equals the exact mode run on
    features rounded here independently and projected by an identity W."""
    rp, ci = G.random_graph(48, 0.15, 8)
    n = len(rp) - 1
    heads, D, F_in = 2, 16, 24
    H = synth.normal_f32((n, F_in), 1.0, 31)
    W = synth.normal_f32((F_in, heads * D), 1.0 / F_in, 32)
    a = synth.normal_f32((heads, D), 1.0 / D, 33)
    # the projection in the oracle's order (k ascending; fp32 products are
    # exact in fp64), so both sides round the very same doubles
    C = np.zeros((n, heads * D), np.float64)
    for k in range(F_in):
        C += H[:, k, None].astype(np.float64) * W[None, k, :].astype(np.float64)
    Cb = _bf16_rne_of_f32(C)
    I = np.zeros((heads * D, heads * D), np.uint16)
    I[np.arange(heads * D), np.arange(heads * D)] = 0x3F80  # bf16 1.0
    ro, rl = oracle.gatv2(rp, ci, H, W, a, heads, D, 0.2, round_c=True)
    eo, el = oracle.gatv2(rp, ci, Cb, I, a, heads, D, 0.2)
    assert np.array_equal(ro, eo) and np.array_equal(rl, el)
    # and it is a different result from the unrounded one
    uo, _ = oracle.gatv2(rp, ci, H, W, a, heads, D, 0.2)
    assert not np.array_equal(uo, ro)
