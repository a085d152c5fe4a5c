"""GPU parity of step a8 (vertex orderings and relabelling) against the CPU
oracle, through the C ABI: every output is compared bit-exactly.  Marked
gpu."""
import numpy as np
import pytest

import oracle
import synth
from tests import graphs as G

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KINDS = [(oracle.PERM_IDENTITY, "identity"), (oracle.PERM_RANDOM, "random"),
         (oracle.PERM_DEGREE, "degree"), (oracle.PERM_RCM, "rcm")]


@pytest.fixture(scope="module")
def gnn():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test was selected but torch sees no CUDA device")
    import sparse_neighbourhood_aggregation_gb300 as m
    m.lib()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_orders(gnn, rp, ci, seed=7):
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    n = len(rp) - 1
    for kind, name in KINDS:
        perm, inv = gnn.gnn_reorder_perm(g, kind, seed)
        ref = oracle.perm(kind, rp, ci, seed=seed)
        p = perm.cpu().numpy()
        assert np.array_equal(p, ref), f"{name} order differs"
        ref_inv = np.empty(n, np.int32)
        ref_inv[ref] = np.arange(n, dtype=np.int32)
        assert np.array_equal(inv.cpu().numpy(), ref_inv), f"{name} inverse differs"


def disconnected(seed=3):
    rng = np.random.default_rng(seed)
    edges = []
    for base, size in [(0, 5), (5, 1), (6, 12), (18, 2), (20, 1), (21, 30)]:
        for _ in range(2 * size):
            a, b = rng.integers(size, size=2)
            edges.append((base + int(a), base + int(b)))
    return G.from_edges(51, edges)


@pytest.mark.parametrize("make", [lambda: G.random_graph(40, 0.08, 1), lambda: G.star(17),
                                  lambda: G.path(33), lambda: G.grid(9), disconnected,
                                  lambda: G.from_edges(12, [], self_loops=True),
                                  lambda: G.from_edges(9, [(1, 2), (2, 1), (7, 3)],
                                                       self_loops=False)])
def test_orders_small_graphs(gnn, make):
    rp, ci = make()
    check_orders(gnn, rp, ci)


def test_orders_shuffled_path_and_grid(gnn):
    for rp, ci in (G.path(200), G.grid(16)):
        n = len(rp) - 1
        p = np.random.default_rng(5).permutation(n).astype(np.int32)
        rp2, ci2 = G.relabel(rp, ci, p)
        check_orders(gnn, rp2, ci2, seed=11)


def test_orders_config1_and_rmat17(gnn):
    for name in ("c1_er1k", "c2_rmat17"):
        w = synth.workload(name, features=False)
        check_orders(gnn, w["rowptr"], w["colidx"])


def test_orders_rmat20(gnn):
    w = synth.workload("c3_rmat20_gatv2", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    for kind, name in KINDS[1:]:
        perm, _ = gnn.gnn_reorder_perm(g, kind, 7)
        assert np.array_equal(perm.cpu().numpy(), oracle.perm(kind, rp, ci, seed=7)), name


def test_apply_perm_graph_and_features(gnn):
    for name in ("c1_er1k", "c2_rmat17"):
        w = synth.workload(name)
        rp, ci, X = w["rowptr"], w["colidx"], w["X"]
        g = gnn.Graph(dev(rp), dev(ci), prepare=False)
        for kind, kname in KINDS:
            p = oracle.perm(kind, rp, ci, seed=7)
            for with_inv in (True, False):
                inv = None
                if with_inv:
                    inv_h = np.empty_like(p)
                    inv_h[p] = np.arange(len(p), dtype=np.int32)
                    inv = dev(inv_h)
                rpo, cio, Xo = gnn.gnn_apply_perm(g, dev(p), inv, X=dev(X))
                rref, cref = oracle.apply_perm(rp, ci, p)
                assert np.array_equal(rpo.cpu().numpy(), rref), f"{name} {kname} rowptr"
                assert np.array_equal(cio.cpu().numpy(), cref), f"{name} {kname} colidx"
                assert np.array_equal(Xo.cpu().numpy(), X[p]), f"{name} {kname} features"
    # bf16 features and an empty graph
    rp, ci = G.from_edges(7, [], self_loops=False)
    g = gnn.Graph(dev(rp), dev(ci), prepare=False)
    Xb = synth.normal_bf16((7, 64), 1.0, 3)
    p = np.array([3, 1, 0, 6, 5, 4, 2], np.int32)
    rpo, cio, Xo = gnn.gnn_apply_perm(g, dev(p),
                                      X=dev(Xb.view(np.int16)).view(torch.bfloat16))
    assert np.array_equal(rpo.cpu().numpy(), np.zeros(8, np.int32))
    assert np.array_equal(Xo.view(torch.int16).cpu().numpy().view(np.uint16), Xb[p])
