"""Small hand-made and random graphs for tests (CSR by destination).

Test helper only: builds inputs, holds no arithmetic of the method."""
import numpy as np


def from_edges(n, edges, self_loops=True):
    """edges: iterable of (src, dst).  Dedupe, optional one self-loop per
    node, CSR by destination with ascending columns."""
    rows = [set() for _ in range(n)]
    for s, d in edges:
        if s != d:
            rows[d].add(int(s))
    if self_loops:
        for i in range(n):
            rows[i].add(i)
    rowptr = np.zeros(n + 1, np.int32)
    cols = []
    for i in range(n):
        r = sorted(rows[i])
        cols.extend(r)
        rowptr[i + 1] = rowptr[i] + len(r)
    return rowptr, np.array(cols, dtype=np.int32)


def random_graph(n, p, seed, self_loops=True):
    rng = np.random.default_rng(seed)
    m = rng.random((n, n)) < p
    edges = [(s, d) for d in range(n) for s in range(n) if m[d, s]]
    return from_edges(n, edges, self_loops)


def star(n, hub=0, self_loops=True):
    return from_edges(n, [(j, hub) for j in range(n) if j != hub] + [(hub, j) for j in range(1, n, 3)],
                      self_loops)


def path(n):
    return from_edges(n, [(i, i + 1) for i in range(n - 1)], True)


def grid(w):
    e = []
    for r in range(w):
        for c in range(w):
            u = r * w + c
            if c + 1 < w:
                e.append((u, u + 1))
            if r + 1 < w:
                e.append((u + w, u))
    return from_edges(w * w, e, True)


def dense_adjacency(rowptr, colidx):
    """Boolean matrix A[i, j] = edge j -> i."""
    n = len(rowptr) - 1
    A = np.zeros((n, n), bool)
    for i in range(n):
        A[i, colidx[rowptr[i]:rowptr[i + 1]]] = True
    return A


def relabel(rowptr, colidx, perm):
    """Relabel by perm (perm[new] = old) with plain Python (test-side):
    edge j -> i becomes inv[j] -> inv[i]; columns re-sorted."""
    n = len(rowptr) - 1
    inv = np.empty(n, np.int64)
    inv[np.asarray(perm)] = np.arange(n)
    rows = [[] for _ in range(n)]
    for i in range(n):
        for j in colidx[rowptr[i]:rowptr[i + 1]]:
            rows[inv[i]].append(int(inv[j]))
    rp = np.zeros(n + 1, np.int32)
    cols = []
    for r in range(n):
        cols.extend(sorted(rows[r]))
        rp[r + 1] = len(cols)
    return rp, np.array(cols, dtype=np.int32)


def read_golden(path):
    d = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = v
    return d
