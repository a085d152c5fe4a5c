"""Segment sum through gnn_segment_reduce_sum_noalloc, the entry point for
callers that cannot allocate device memory (a plugin whose host framework
owns every allocation, or a loop that cannot afford cudaMalloc's implicit
synchronisation): its scratch is a fixed library-owned device array instead
of a caller workspace.

The test calls it through the C ABI twice in a row and compares each result
with gnn_segment_reduce_sum (the workspace entry point) on the same input.
The graphs carry rows longer than one edge run, so the partial sums and
arrival counters held in the fixed array are used; the second call shows
that leftovers from the first do not leak into it.  The file is named to be
collected last.  Marked gpu."""
import ctypes

import numpy as np
import pytest

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _hub_graph(n, hubs, deg, seed):
    rng = np.random.default_rng(seed)
    edges = [(int(s), h) for h in hubs for s in rng.choice(n, deg, replace=False)]
    edges += [(int(rng.integers(n)), int(rng.integers(n))) for _ in range(4 * n)]
    return G.from_edges(n, edges)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_matches_workspace_entry_point_twice(gnn, dtype):
    rp, ci = _hub_graph(3000, (0, 17, 2999), 2500, 5)
    n = len(rp) - 1
    if dtype == "f32":
        X, tol = _dev(synth.normal_f32((n, 128), 1.0, 21)), TOL_F32
    else:
        bits = synth.normal_bf16((n, 256), 1.0, 21)
        X, tol = _dev(bits.view(np.int16)).view(torch.bfloat16), TOL_BF16
    g = gnn.graph_prepare(_dev(rp), _dev(ci))
    need = gnn.lib().gnn_workspace_size(gnn.GNN_OP_SUM, ctypes.byref(g.csr), X.shape[1], 0, 0)
    assert need <= 8 << 20
    ref = gnn.gnn_segment_reduce_sum(g, X).cpu().numpy()
    for _ in range(2):
        Y = torch.full((n, X.shape[1]), float("nan"), device="cuda")
        gnn.gnn_segment_reduce_sum_noalloc(g, X, out=Y)
        torch.cuda.synchronize()
        assert_rowwise_close(Y.cpu().numpy(), ref, tol, f"noalloc sum {dtype}")


def test_noalloc_without_prepared_graph(gnn):
    rp, ci = _hub_graph(1200, (7,), 1100, 6)
    n = len(rp) - 1
    X = _dev(synth.normal_f32((n, 64), 1.0, 22))
    g = gnn.Graph(_dev(rp), _dev(ci), prepare=False)
    ref = gnn.gnn_segment_reduce_sum(g, X).cpu().numpy()
    for _ in range(2):
        Y = gnn.gnn_segment_reduce_sum_noalloc(g, X).cpu().numpy()
        assert_rowwise_close(Y, ref, TOL_F32, "noalloc sum, no prep")


def test_noalloc_rejects_problems_beyond_the_fixed_scratch(gnn):
    b = gnn
    # 4M edges at F = 128 need ~32 MB of scratch: refused on the host,
    # before any launch (the pointers below are never dereferenced)
    csr = b.binding.gnn_csr(1 << 20, 1 << 20, 4 << 20, 256, 256, None)
    rc = b.lib().gnn_segment_reduce_sum_noalloc(ctypes.byref(csr), None, 256, b.GNN_F32, 128,
                                                256, None)
    assert rc == b.GNN_ERR_WORKSPACE


def test_noalloc_rejections_match_the_workspace_entry_point(gnn):
    """A call refused on the host returns gnn_segment_reduce_sum's code and
    launches nothing, so the shared array and the stream are untouched: a
    valid call right after it still matches the workspace entry point."""
    rp, ci = _hub_graph(2000, (3, 1500), 1800, 7)
    n = len(rp) - 1
    X = _dev(synth.normal_f32((n, 128), 1.0, 23))
    g = gnn.graph_prepare(_dev(rp), _dev(ci))
    L = gnn.lib()
    ws = g.workspace(gnn.GNN_OP_SUM, 128)
    Y = torch.zeros((n, 128), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    prep = g.prep.data_ptr()
    cases = [
        # F = 6 is not a whole number of 16-byte fp32 chunks
        dict(F=6, Y=Y.data_ptr(), dt=gnn.GNN_F32),
        # no output buffer
        dict(F=128, Y=None, dt=gnn.GNN_F32),
        # an unknown dtype code
        dict(F=128, Y=Y.data_ptr(), dt=7),
        # a negative width
        dict(F=-128, Y=Y.data_ptr(), dt=gnn.GNN_F32),
    ]
    for c in cases:
        ref_rc = L.gnn_segment_reduce_sum(ctypes.byref(g.csr), prep, X.data_ptr(), c["dt"],
                                          c["F"], c["Y"], ws.data_ptr(), ws.numel(), stream)
        rc = L.gnn_segment_reduce_sum_noalloc(ctypes.byref(g.csr), prep, X.data_ptr(), c["dt"],
                                              c["F"], c["Y"], stream)
        assert ref_rc != gnn.GNN_OK, c
        assert rc == ref_rc, (c, rc, ref_rc)
    ref = gnn.gnn_segment_reduce_sum(g, X).cpu().numpy()
    got = gnn.gnn_segment_reduce_sum_noalloc(g, X).cpu().numpy()
    assert_rowwise_close(got, ref, TOL_F32, "noalloc sum after refused calls")
