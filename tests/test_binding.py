"""The Python binding has no CPU path: without the built library it raises,
and CPU tensors are refused before any call.  CPU only."""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_raises():
    code = ("import sparse_neighbourhood_aggregation_gb300 as g\n"
            "try:\n    g.lib()\nexcept RuntimeError as e:\n    print('raised:', e)\n")
    env = dict(os.environ, GNN_LIB_PATH=os.path.join(ROOT, "no_such_dir", "libgnn.so"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.startswith("raised:") and "not built" in r.stdout


def test_cpu_tensors_are_refused():
    import sparse_neighbourhood_aggregation_gb300 as g
    rp = torch.tensor([0, 1, 2], dtype=torch.int32)
    ci = torch.tensor([0, 1], dtype=torch.int32)
    with pytest.raises(ValueError):
        g.Graph(rp, ci)
    x = torch.from_numpy(np.zeros((2, 32), np.float32))
    with pytest.raises(ValueError):
        g.gnn_projection(x, torch.zeros((32, 32)))
