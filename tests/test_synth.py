"""The seeded input generators: CSR structure (ascending unique columns, one
self-loop per node), determinism, the recorded workload sizes, the degree
and cluster structure the recipes promise, and the value distributions.
CPU only."""
import numpy as np
import pytest

import synth


def check_csr(rp, ci, n):
    assert rp.dtype == np.int32 and ci.dtype == np.int32
    assert len(rp) == n + 1 and rp[0] == 0 and rp[-1] == len(ci)
    assert np.all(np.diff(rp) >= 0)
    assert ci.min() >= 0 and ci.max() < n
    rows = np.repeat(np.arange(n), np.diff(rp))
    # ascending and unique within each row
    same_row = rows[1:] == rows[:-1]
    assert np.all(ci[1:][same_row] > ci[:-1][same_row])
    # exactly one self-loop per node
    loops = ci == rows
    assert loops.sum() == n and np.array_equal(np.sort(rows[loops]), np.arange(n))


def test_er_structure_and_size():
    rp, ci = synth.er(1024, 8192)
    check_csr(rp, ci, 1024)
    assert len(ci) == 8192 + 1024  # distinct non-loop edges plus the loops


@pytest.mark.parametrize("scale", [10, 12])
def test_rmat_structure_and_power_law(scale):
    rp, ci = synth.rmat(scale, 16, *synth.RMAT_ABC)
    n = 1 << scale
    check_csr(rp, ci, n)
    deg = np.diff(rp)
    # duplicates removed: fewer than edge factor x n draws plus the loops
    assert n < len(ci) <= 16 * n + n
    # heavy tail, growing with the scale
    top = np.sort(deg)[::-1][: int(0.06 * n)]
    assert top.sum() > 0.4 * len(ci)
    assert deg.max() > 20 * deg.mean()


def test_rmat17_size_and_shape_are_the_recorded_ones():
    """R-MAT scale 17 as recorded: 2,074,264 edges; the shape of the
    power-law workloads: the top 6% of rows hold about 70% of the edges,
    about 41% of the nodes have only their self-loop, the largest in-degree
    is about 10K."""
    w = synth.workload("c2_rmat17", features=False)
    rp, ci = w["rowptr"], w["colidx"]
    n = 1 << 17
    assert len(ci) == 2_074_264
    check_csr(rp, ci, n)
    deg = np.diff(rp)
    assert 0.65 < np.sort(deg)[::-1][: int(0.06 * n)].sum() / len(ci) < 0.75
    assert 0.38 < (deg == 1).mean() < 0.44
    assert 8_000 < deg.max() < 12_000


def test_generators_are_deterministic():
    a = synth.rmat(11, 16, *synth.RMAT_ABC)
    b = synth.rmat(11, 16, *synth.RMAT_ABC)
    c = synth.rmat(11, 16, *synth.RMAT_ABC, seed=synth.SEED_GRAPH + 1)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[1], c[1])
    assert np.array_equal(synth.normal_f32((64, 8), 1.0, 3), synth.normal_f32((64, 8), 1.0, 3))
    assert not np.array_equal(synth.normal_f32((64, 8), 1.0, 3), synth.normal_f32((64, 8), 1.0, 4))


def test_clustered_structure():
    n_c, size, p, rewire = 16, 128, 0.3, 0.05
    rp, ci = synth.clustered(n_c, size, p, rewire, 7)
    n = n_c * size
    check_csr(rp, ci, n)
    rows = np.repeat(np.arange(n), np.diff(rp))
    off = ci != rows
    inside = (ci[off] // size) == (rows[off] // size)
    # a fraction `rewire` of the non-loop edges leave their cluster (a
    # rewired source can land in its own cluster with probability 1/n_c)
    frac_out = 1.0 - inside.mean()
    assert abs(frac_out - rewire * (1 - 1 / n_c)) < 0.01
    # intra-cluster density near p
    dens = inside.sum() / (n_c * size * (size - 1))
    assert abs(dens - p * (1 - rewire)) < 0.02


def test_value_distributions():
    x = synth.normal_f32((200_000,), 0.25, 5)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 0.25) < 0.01
    u = synth.uniform_f32((200_000,), -1.0, 1.0, 6)
    assert u.min() >= -1.0 and u.max() <= 1.0 and abs(u.var() - 1 / 3) < 0.01
    bits = synth.normal_bf16((200_000,), 1.0, 5)
    f = synth.bf16_to_f32(bits)
    assert abs(f.var() - 1.0) < 0.02
    # bf16 is round-to-nearest-even of the same fp32 draw
    x1 = synth.normal_f32((4096,), 1.0, 8)
    b1 = synth.bf16_to_f32(synth.normal_bf16((4096,), 1.0, 8))
    u32 = x1.view(np.uint32).astype(np.uint64)
    rne = ((u32 + 0x7FFF + ((u32 >> 16) & 1)) >> 16).astype(np.uint32) << 16
    assert np.array_equal(b1.view(np.uint32), rne.astype(np.uint32))
