"""GB300-native CSR neighbourhood aggregation for GNN layers.

The compute lives in libgnn.so (C ABI, include/gnn.h; hand-written CUDA for
sm_103a).  This package is its thin Python binding; PyTorch provides device
memory and streams only.
"""
from .binding import *  # noqa: F401,F403
from .binding import Graph, GnnError, graph_prepare, lib  # noqa: F401

__all__ = [n for n in dir() if n.startswith("gnn_") or n.startswith("GNN_")] + [
    "Graph", "GnnError", "graph_prepare", "lib", "csr_validate", "launch_count", "version"]
