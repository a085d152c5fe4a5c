"""Host-side logic of bench.py (no GPU): the recorded-traffic lookup that
ties an ncu DRAM figure to the kernel sources it was captured on, the
whole-job rate, and the bounded row sample of the CPU baseline."""
import numpy as np

import bench


def _table(tmp_path, rows):
    p = tmp_path / "dram_traffic.md"
    lines = ["| workload | layer | dram bytes per layer call | sources sha16 | capture |",
             "|---|---|---|---|---|"]
    lines += [f"| {w} | {l} | {b} | {h} | test |" for w, l, b, h in rows]
    p.write_text("\n".join(lines) + "\n")
    return str(p)


def test_recorded_traffic_needs_the_sources_hash(tmp_path, monkeypatch):
    sha = bench.sources_sha16(bench.TRAFFIC_SOURCES["spmm"])
    monkeypatch.setattr(bench, "TRAFFIC_TABLE", _table(tmp_path, [
        ("c5_rmat22", "spmm", 123456, sha),
        ("c2_rmat17", "sum", 777, "0000000000000000"),
    ]))
    assert bench.recorded_traffic("c5_rmat22", "spmm") == (123456.0, sha)
    # a capture of other kernel sources is stale: no figure, the current hash
    assert bench.recorded_traffic("c2_rmat17", "sum") == (None, sha)
    # no row, or a layer without recorded sources
    assert bench.recorded_traffic("c2_rmat17", "mean") == (None, sha)
    assert bench.recorded_traffic("c5_rmat22", "gatv2_fwd") == (None, None)


def test_sources_hash_follows_the_file_contents(tmp_path, monkeypatch):
    for name, text in (("a.cu", "x"), ("b.cuh", "y")):
        (tmp_path / name).write_text(text)
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    h0 = bench.sources_sha16(("a.cu", "b.cuh"))
    assert len(h0) == 16 and h0 == bench.sources_sha16(("a.cu", "b.cuh"))
    (tmp_path / "b.cuh").write_text("y ")
    assert bench.sources_sha16(("a.cu", "b.cuh")) != h0


def test_committed_traffic_table_parses():
    # every data row of the committed table carries an integer byte count
    # and a 16-digit hash
    with open(bench.TRAFFIC_TABLE) as f:
        rows = [[c.strip() for c in ln.strip().strip("|").split("|")] for ln in f
                if ln.startswith("| c")]
    assert rows
    for r in rows:
        assert int(r[2]) > 0 and len(r[3]) == 16 and int(r[3], 16) >= 0


def test_job_rate_is_units_over_time():
    # 2 ranks x 1e9 units a step x 10 steps in 4 s = 5 G units/s
    assert bench.job_rate(2, 1e9, 10, 4000.0) == 5.0


def test_sample_by_edges_is_bounded_and_sorted():
    rng = np.random.default_rng(3)
    deg = rng.integers(0, 40, size=5000)
    rp = np.concatenate([[0], np.cumsum(deg)]).astype(np.int32)
    rows, edges = bench._sample_by_edges(rp, 20000)
    assert np.all(np.diff(rows) > 0)
    assert edges == int(np.sum(deg[rows]))
    assert 20000 <= edges < 20000 + 40
    assert bench._sample_by_edges(rp, 20000)[0].tolist() == rows.tolist()
