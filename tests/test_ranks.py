"""The bench's multi-rank host logic on CPU: world-size-2 gloo ranks take
the slowest rank's time and report the whole job's units, and the reference
arm runs on rank 0 alone.  CPU only."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = bench.max_over_ranks(torch, 10.0 + 5.0 * rank, world)  # rank 1 is the slow one
    out[rank] = (ms, bench.job_rate(world, 1e6, 4, ms))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        want = (15.0, 2 * 1e6 * 4 / 15e-3 / 1e9)
        assert out[0] == pytest.approx(want) and out[1] == pytest.approx(want)


def test_one_rank_keeps_its_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(torch, 7.5, 1) == 7.5
    assert bench.job_rate(1, 2e9, 3, 1000.0) == pytest.approx(6.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.strip() == ""
