// Step a8: vertex orderings (identity, random, degree, reverse Cuthill-McKee)
// and the relabelling of a CSR graph and its feature rows.
//
// IO-aware GNN layers, Section 2.4 and Section 4.1 (graph reordering as a
// cache-locality lever whose benefit depends on the kernel mapping); RCM as
// named in "A High-Throughput Solver for Marginalized Graph Kernels on GPU"
// (graph reordering section).  The orders are defined exactly so that one
// answer is correct (ties by node id), and every output here is bit-exact.
//
// GB300 design.  Every step is a device kernel or a device-wide sort / scan
// (CUB radix sort and scan, compiled into this library); the host only
// sequences the breadth-first levels of RCM.
//  * RANDOM: key splitmix64(seed ^ id) (Steele, Lea, Flood 2014), stable
//    radix sort of (key, id) -> ascending (key, id).
//  * DEGREE: key ~(d_in + d_out) (as stored), stable radix sort -> descending
//    total degree, ties by ascending id.
//  * RCM on S = A + A^T without self-loops.  Sequential Cuthill-McKee is
//    reproduced level-synchronously: (1) connected components (hook to the
//    smaller root with atomicMin + pointer shortcutting); (2) each
//    component's breadth-first search starts at its own smallest
//    (degree, id) node, and components are laid out in the order of those
//    start keys -- exactly the order in which the sequential method starts
//    them, since it always starts at the smallest unvisited key; (3) all
//    components advance one level at a time; a node reached at level L+1
//    takes as parent its earliest-placed neighbour at level L (atomicMin of
//    positions), which is the neighbour whose dequeue appends it in the
//    sequential method; the level is ordered by (parent position, degree,
//    id) with one radix sort and placed after the component's previous
//    levels.  The sequence is reversed at the end.
//  * apply_perm: one radix sort of the 64-bit keys (new row << 32 | new
//    column) yields the relabelled CSR with columns ascending in every row.
#include <cub/device/device_radix_sort.cuh>
#include <cub/device/device_scan.cuh>

#include <algorithm>
#include <vector>

#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);

namespace {

// SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): the output function applied to state x.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int bits_for(int64_t v) {
    int b = 1;
    while (b < 63 && ((int64_t)1 << b) <= v) ++b;
    return b;
}

__global__ void k_iota(int32_t *__restrict__ out, int32_t n) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = i;
}

__global__ void k_random_keys(uint64_t *__restrict__ key, int32_t *__restrict__ id, int32_t n, uint64_t seed) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        key[i] = splitmix64(seed ^ (uint64_t)i);
        id[i] = i;
    }
}

// key = ~(d_in + d_out) so that an ascending sort is descending degree
__global__ void k_degree_keys(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ d_out,
                              uint32_t *__restrict__ key, int32_t *__restrict__ id, int32_t n) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const uint32_t d = (uint32_t)(rowptr[i + 1] - rowptr[i]) + (uint32_t)d_out[i];
        key[i] = ~d;
        id[i] = i;
    }
}

__global__ void k_count_cols(const int32_t *__restrict__ colidx, int64_t nnz, int32_t *__restrict__ cnt) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride)
        atomicAdd(&cnt[colidx[e]], 1);
}

// row id of every edge (one warp per row, lanes over its edges)
__global__ void k_edge_rows(const int32_t *__restrict__ rowptr, int32_t n, int32_t *__restrict__ rowid) {
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= n) return;
    const int32_t b = rowptr[wid], e = rowptr[wid + 1];
    for (int32_t k = b + lane; k < e; k += 32) rowid[k] = (int32_t)wid;
}

// inv[perm[i]] = i
__global__ void k_inv_from_perm(const int32_t *__restrict__ perm, int32_t *__restrict__ inv, int32_t n) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) inv[perm[i]] = i;
}

// |S(i)|, S = A + A^T without self-loops: the distinct ids other than i in
// the sorted row i of A and row i of A^T.  A thread merges the two lists of a
// row whose lengths sum to at most kSymLight; longer rows are queued for
// k_sym_degree_heavy (heavy[0..*n_heavy)).
constexpr int32_t kSymLight = 1024;

__global__ void k_sym_degree(const int32_t *__restrict__ rp, const int32_t *__restrict__ ci,
                             const int32_t *__restrict__ tp, const int32_t *__restrict__ tc, int32_t n,
                             int32_t *__restrict__ sdeg, int32_t *__restrict__ heavy, int32_t *n_heavy) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    int32_t a = rp[i], ae = rp[i + 1], b = tp[i], be = tp[i + 1];
    if ((ae - a) + (be - b) > kSymLight) {
        heavy[atomicAdd(n_heavy, 1)] = i;
        return;
    }
    int32_t cnt = 0;
    while (a < ae || b < be) {
        int32_t x;
        if (b >= be || (a < ae && ci[a] < tc[b])) x = ci[a++];
        else if (a >= ae || tc[b] < ci[a]) x = tc[b++];
        else { x = ci[a++]; ++b; }
        cnt += (x != i);
    }
    sdeg[i] = cnt;
}

// first position in sorted v[lo, hi) holding a value >= x
__device__ __forceinline__ int32_t lower_bound_i32(const int32_t *__restrict__ v, int32_t lo, int32_t hi,
                                                   int32_t x) {
    while (lo < hi) {
        const int32_t mid = lo + ((hi - lo) >> 1);
        if (v[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// A block per queued row: |S(i)| = |P \ {i}| + |Q \ {i}| - |(P n Q) \ {i}|,
// P the shorter of the two lists; each thread takes every blockDim-th
// element of P and looks it up in Q by binary search.  Exact integer counts.
__global__ void __launch_bounds__(256) k_sym_degree_heavy(const int32_t *__restrict__ rp,
                                                          const int32_t *__restrict__ ci,
                                                          const int32_t *__restrict__ tp,
                                                          const int32_t *__restrict__ tc,
                                                          const int32_t *__restrict__ heavy,
                                                          const int32_t *n_heavy, int32_t *__restrict__ sdeg) {
    __shared__ int32_t s_inter, s_self_p, s_self_q;
    const int32_t nh = *n_heavy;
    for (int32_t q = blockIdx.x; q < nh; q += gridDim.x) {
        const int32_t i = heavy[q];
        const int32_t *P = ci + rp[i], *Q = tc + tp[i];
        int32_t np = rp[i + 1] - rp[i], nq = tp[i + 1] - tp[i];
        if (np > nq) {
            const int32_t *t = P; P = Q; Q = t;
            const int32_t tn = np; np = nq; nq = tn;
        }
        if (threadIdx.x == 0) {
            s_inter = 0;
            s_self_p = 0;
            const int32_t k = lower_bound_i32(Q, 0, nq, i);
            s_self_q = (k < nq && Q[k] == i) ? 1 : 0;
        }
        __syncthreads();
        int32_t inter = 0, self_p = 0;
        for (int32_t k = threadIdx.x; k < np; k += blockDim.x) {
            const int32_t x = P[k];
            if (x == i) { self_p = 1; continue; }
            const int32_t j = lower_bound_i32(Q, 0, nq, x);
            inter += (j < nq && Q[j] == x) ? 1 : 0;
        }
        if (inter) atomicAdd(&s_inter, inter);
        if (self_p) atomicAdd(&s_self_p, 1);
        __syncthreads();
        if (threadIdx.x == 0) sdeg[i] = (np - s_self_p) + (nq - s_self_q) - s_inter;
        __syncthreads();
    }
}

// connected components of A (direction ignored): hook roots to the smaller
// root; parent pointers only ever decrease, so no cycle can form.  Reads go
// to L2 (other blocks update the pointers with atomics during the pass).
__device__ __forceinline__ int32_t cc_find(const int32_t *parent, int32_t v) {
    int32_t p = __ldcg(parent + v);
    while (p != v) {
        v = p;
        p = __ldcg(parent + v);
    }
    return v;
}

__global__ void k_cc_hook(const int32_t *__restrict__ rowid, const int32_t *__restrict__ colidx, int64_t nnz,
                          int32_t *parent, int32_t *changed) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) {
        int32_t ru = cc_find(parent, rowid[e]), rv = cc_find(parent, colidx[e]);
        if (ru == rv) continue;
        const int32_t hi = max(ru, rv), lo = min(ru, rv);
        atomicMin(&parent[hi], lo);
        *changed = 1;
    }
}

__global__ void k_cc_shortcut(int32_t *parent, int32_t n) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) parent[i] = cc_find(parent, i);
}

// component of every node = its root (the component's smallest id);
// per root: smallest (degree, id) rank and size
__global__ void k_comp_stats(const int32_t *__restrict__ root, const int32_t *__restrict__ rank, int32_t n,
                             int32_t *__restrict__ comp_min_rank, int32_t *__restrict__ comp_size) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    atomicMin(&comp_min_rank[root[i]], rank[i]);
    atomicAdd(&comp_size[root[i]], 1);
}

// size_by_rank[k] = size of the component whose smallest rank is k (else 0)
__global__ void k_size_by_rank(const int32_t *__restrict__ root, const int32_t *__restrict__ comp_min_rank,
                               const int32_t *__restrict__ comp_size, int32_t n, int32_t *__restrict__ by_rank) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n && root[i] == i) by_rank[comp_min_rank[i]] = comp_size[i];
}

// level 0: every component's start node takes the component's first
// position; fill[root] = next free position of the component
__global__ void k_bfs_start(const int32_t *__restrict__ root, const int32_t *__restrict__ comp_min_rank,
                            const int32_t *__restrict__ base_by_rank, const int32_t *__restrict__ order_di,
                            int32_t n, int32_t *__restrict__ pos, int32_t *__restrict__ fill,
                            int32_t *__restrict__ frontier, int32_t *__restrict__ nfront) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n || root[i] != i) return;
    const int32_t r = comp_min_rank[i];
    const int32_t s = order_di[r];
    const int32_t b = base_by_rank[r];
    pos[s] = b;
    fill[i] = b + 1;
    frontier[atomicAdd(nfront, 1)] = s;
}

// expand one level: neighbours v of frontier nodes u (in S, v != u) that
// have no position yet take the smallest parent position and are listed once
__global__ void k_bfs_expand(const int32_t *__restrict__ rp, const int32_t *__restrict__ ci,
                             const int32_t *__restrict__ tp, const int32_t *__restrict__ tc,
                             const int32_t *__restrict__ frontier, int32_t nfront,
                             const int32_t *__restrict__ pos, int32_t *__restrict__ ppos,
                             int32_t *__restrict__ flag, int32_t *__restrict__ cand, int32_t *__restrict__ ncand) {
    const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= nfront) return;
    const int32_t u = frontier[wid];
    const int32_t pu = pos[u];
    for (int side = 0; side < 2; ++side) {
        const int32_t *p = side ? tp : rp;
        const int32_t *c = side ? tc : ci;
        const int32_t b = p[u], e = p[u + 1];
        for (int32_t k = b + lane; k < e; k += 32) {
            const int32_t v = c[k];
            if (v == u || pos[v] >= 0) continue;
            atomicMin(&ppos[v], pu);
            if (atomicExch(&flag[v], 1) == 0) cand[atomicAdd(ncand, 1)] = v;
        }
    }
}

__global__ void k_level_keys(const int32_t *__restrict__ cand, int32_t nc, const int32_t *__restrict__ ppos,
                             const int32_t *__restrict__ rank, uint64_t *__restrict__ key) {
    const int32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < nc) {
        const int32_t v = cand[k];
        key[k] = ((uint64_t)(uint32_t)ppos[v] << 32) | (uint32_t)rank[v];
    }
}

// start index of the component segment each sorted candidate falls in
__global__ void k_seg_heads(const int32_t *__restrict__ sorted, int32_t nc, const int32_t *__restrict__ root,
                            int32_t *__restrict__ head) {
    const int32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < nc) head[k] = (k == 0 || root[sorted[k]] != root[sorted[k - 1]]) ? k : 0;
}

struct MaxOp {
    __device__ __forceinline__ int32_t operator()(int32_t a, int32_t b) const { return a > b ? a : b; }
};

__global__ void k_level_place(const int32_t *__restrict__ sorted, int32_t nc, const int32_t *__restrict__ root,
                              const int32_t *__restrict__ seg, const int32_t *__restrict__ fill,
                              int32_t *__restrict__ pos) {
    const int32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < nc) {
        const int32_t v = sorted[k];
        pos[v] = fill[root[v]] + (k - seg[k]);
    }
}

__global__ void k_level_fill(const int32_t *__restrict__ sorted, int32_t nc, const int32_t *__restrict__ root,
                             const int32_t *__restrict__ pos, int32_t *__restrict__ fill) {
    const int32_t k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k < nc && (k == nc - 1 || root[sorted[k]] != root[sorted[k + 1]])) {
        const int32_t v = sorted[k];
        fill[root[v]] = pos[v] + 1;
    }
}

// perm[new] = the node at position n-1-new (the reversal of the sequence)
__global__ void k_rcm_emit(const int32_t *__restrict__ pos, int32_t n, int32_t *__restrict__ perm) {
    const int32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (v < n) perm[n - 1 - pos[v]] = v;
}

__global__ void k_fill_i32(int32_t *__restrict__ p, int32_t n, int32_t v) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = v;
}

// ---------------------------------------------------------------- apply_perm

__global__ void k_new_degrees(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ perm, int32_t n,
                              int32_t *__restrict__ deg) {
    const int32_t r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < n) deg[r] = rowptr[perm[r] + 1] - rowptr[perm[r]];
    if (r == n) deg[r] = 0;
}

// keys (new row << 32 | new column) of every edge, new row r taking old row
// perm[r] (one warp per row)
__global__ void k_relabel_keys(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ colidx,
                               const int32_t *__restrict__ perm, const int32_t *__restrict__ inv,
                               const int32_t *__restrict__ rowptr_out, int32_t n, uint64_t *__restrict__ key) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= n) return;
    const int32_t o = perm[r];
    const int32_t b = rowptr[o], d = rowptr[o + 1] - b, ob = rowptr_out[r];
    for (int32_t k = lane; k < d; k += 32)
        key[ob + k] = ((uint64_t)r << 32) | (uint32_t)inv[colidx[b + k]];
}

__global__ void k_low_words(const uint64_t *__restrict__ key, int64_t m, int32_t *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < m; e += stride)
        out[e] = (int32_t)(uint32_t)key[e];
}

// X_out[r] = X[perm[r]] (rows of row_bytes, a multiple of 16; warp per row)
__global__ void k_gather_rows(const uint4 *__restrict__ X, const int32_t *__restrict__ perm, int32_t n,
                              int64_t row_chunks, uint4 *__restrict__ Y) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= n) return;
    const uint4 *src = X + (int64_t)perm[r] * row_chunks;
    uint4 *dst = Y + r * row_chunks;
    for (int64_t c = lane; c < row_chunks; c += 32) dst[c] = src[c];
}

int blocks_for(int64_t n, int t = 256) { return (int)std::max<int64_t>(1, (n + t - 1) / t); }

// ------------------------------------------------------------ workspace

struct ReorderWs {
    // shared by all kinds
    uint64_t *key64[2];
    uint32_t *key32[2];
    int32_t *id[2];
    int32_t *dout;
    // RCM
    int32_t *tp, *tc, *rowid, *tkeys;  // A^T rowptr / colidx, edge row ids, sorted column keys
    int32_t *sdeg, *order_di, *rank, *parent, *cmin, *csize, *by_rank, *base;
    int32_t *pos, *ppos, *flag, *fill, *front, *cand, *seg;
    int32_t *counters;                 // [0] changed, [1] frontier size, [2] candidate count, [3] heavy rows
    void *temp;
    size_t temp_bytes;
    size_t bytes;
};

size_t cub_temp_bytes(int32_t n, int64_t m) {
    size_t t = 0, x = 0;
    cub::DeviceRadixSort::SortPairs(nullptr, x, (const uint64_t *)nullptr, (uint64_t *)nullptr,
                                    (const int32_t *)nullptr, (int32_t *)nullptr, n);
    t = std::max(t, x);
    cub::DeviceRadixSort::SortPairs(nullptr, x, (const uint32_t *)nullptr, (uint32_t *)nullptr,
                                    (const int32_t *)nullptr, (int32_t *)nullptr, std::max<int64_t>(n, m));
    t = std::max(t, x);
    cub::DeviceRadixSort::SortKeys(nullptr, x, (const uint64_t *)nullptr, (uint64_t *)nullptr, m);
    t = std::max(t, x);
    cub::DeviceScan::ExclusiveSum(nullptr, x, (const int32_t *)nullptr, (int32_t *)nullptr, n + 1);
    t = std::max(t, x);
    cub::DeviceScan::InclusiveScan(nullptr, x, (const int32_t *)nullptr, (int32_t *)nullptr, MaxOp(), n);
    t = std::max(t, x);
    return t;
}

ReorderWs reorder_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    ReorderWs W;
    const int32_t n = g->n_rows;
    const int64_t m = g->nnz;
    for (int k = 0; k < 2; ++k) {
        W.key64[k] = c.take<uint64_t>(n);
        W.key32[k] = c.take<uint32_t>(n);
        W.id[k] = c.take<int32_t>(n);
    }
    W.dout = c.take<int32_t>(n + 1);
    W.tp = c.take<int32_t>(n + 1);
    W.tc = c.take<int32_t>(m);
    W.rowid = c.take<int32_t>(m);
    W.tkeys = c.take<int32_t>(m);
    W.sdeg = c.take<int32_t>(n);
    W.order_di = c.take<int32_t>(n);
    W.rank = c.take<int32_t>(n);
    W.parent = c.take<int32_t>(n);
    W.cmin = c.take<int32_t>(n);
    W.csize = c.take<int32_t>(n);
    W.by_rank = c.take<int32_t>(n + 1);
    W.base = c.take<int32_t>(n + 1);
    W.pos = c.take<int32_t>(n);
    W.ppos = c.take<int32_t>(n);
    W.flag = c.take<int32_t>(n);
    W.fill = c.take<int32_t>(n);
    W.front = c.take<int32_t>(n);
    W.cand = c.take<int32_t>(n);
    W.seg = c.take<int32_t>(n);
    W.counters = c.take<int32_t>(4);
    W.temp_bytes = cub_temp_bytes(n, m);
    W.temp = c.take<char>(W.temp_bytes);
    W.bytes = c.used;
    return W;
}

struct PermWs {
    uint64_t *key[2];
    int32_t *deg, *inv;
    void *temp;
    size_t temp_bytes;
    size_t bytes;
};

PermWs perm_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    PermWs W;
    const int32_t n = g->n_rows;
    const int64_t m = g->nnz;
    W.key[0] = c.take<uint64_t>(m);
    W.key[1] = c.take<uint64_t>(m);
    W.deg = c.take<int32_t>(n + 1);
    W.inv = c.take<int32_t>(n);
    W.temp_bytes = cub_temp_bytes(n, m);
    W.temp = c.take<char>(W.temp_bytes);
    W.bytes = c.used;
    return W;
}

#define GNN_CUDA_TRY(x)                                       \
    do {                                                      \
        cudaError_t e__ = (x);                                \
        if (e__ != cudaSuccess) return ::gnn::cuda_status(e__); \
    } while (0)

gnn_status rcm_order(const gnn_csr *g, ReorderWs &W, int32_t *perm, cudaStream_t s) {
    const int32_t n = g->n_rows;
    const int64_t m = g->nnz;
    const int bn = bits_for(n);
    size_t tb = W.temp_bytes;
    // A^T: stable sort of (source, destination) by source
    GNN_CUDA_TRY(cudaMemsetAsync(W.dout, 0, sizeof(int32_t) * (n + 1), s));
    if (m > 0) {
        k_count_cols<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(g->colidx, m, W.dout);
        k_edge_rows<<<blocks_for((int64_t)n * 32), 256, 0, s>>>(g->rowptr, n, W.rowid);
        note_launch(2);
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, g->colidx, W.tkeys, W.rowid, W.tc, m, 0, bn, s));
        note_launch();
    }
    GNN_CUDA_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.dout, W.tp, n + 1, s));
    note_launch();
    // degrees in S and the (degree, id) ranks
    // (cmin is free until the components pass: it holds the queued heavy rows)
    GNN_CUDA_TRY(cudaMemsetAsync(W.counters + 3, 0, sizeof(int32_t), s));
    k_sym_degree<<<blocks_for(n), 256, 0, s>>>(g->rowptr, g->colidx, W.tp, W.tc, n, W.sdeg, W.cmin,
                                                W.counters + 3);
    k_sym_degree_heavy<<<sm_count() * 4, 256, 0, s>>>(g->rowptr, g->colidx, W.tp, W.tc, W.cmin, W.counters + 3,
                                                      W.sdeg);
    k_iota<<<blocks_for(n), 256, 0, s>>>(W.id[0], n);
    note_launch(3);
    GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, reinterpret_cast<const uint32_t *>(W.sdeg),
                                                 W.key32[1], W.id[0], W.order_di, n, 0, 32, s));
    note_launch();
    k_inv_from_perm<<<blocks_for(n), 256, 0, s>>>(W.order_di, W.rank, n);
    // connected components
    k_iota<<<blocks_for(n), 256, 0, s>>>(W.parent, n);
    note_launch(2);
    for (int it = 0; it < 64; ++it) {
        int32_t changed = 0;
        GNN_CUDA_TRY(cudaMemsetAsync(W.counters, 0, sizeof(int32_t), s));
        if (m > 0) {
            k_cc_hook<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(W.rowid, g->colidx, m, W.parent,
                                                                              W.counters);
            note_launch();
        }
        k_cc_shortcut<<<blocks_for(n), 256, 0, s>>>(W.parent, n);
        note_launch();
        GNN_CUDA_TRY(cudaMemcpyAsync(&changed, W.counters, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
        GNN_CUDA_TRY(cudaStreamSynchronize(s));
        if (!changed) break;
        if (it == 63) return GNN_ERR_TIMEOUT;
    }
    // components: start rank, size, base position in start-key order
    k_fill_i32<<<blocks_for(n), 256, 0, s>>>(W.cmin, n, INT32_MAX);
    note_launch();
    GNN_CUDA_TRY(cudaMemsetAsync(W.csize, 0, sizeof(int32_t) * n, s));
    GNN_CUDA_TRY(cudaMemsetAsync(W.by_rank, 0, sizeof(int32_t) * (n + 1), s));
    k_comp_stats<<<blocks_for(n), 256, 0, s>>>(W.parent, W.rank, n, W.cmin, W.csize);
    k_size_by_rank<<<blocks_for(n), 256, 0, s>>>(W.parent, W.cmin, W.csize, n, W.by_rank);
    note_launch(2);
    GNN_CUDA_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.by_rank, W.base, n + 1, s));
    note_launch();
    // breadth-first levels of all components together
    k_fill_i32<<<blocks_for(n), 256, 0, s>>>(W.pos, n, -1);
    k_fill_i32<<<blocks_for(n), 256, 0, s>>>(W.ppos, n, INT32_MAX);
    note_launch(2);
    GNN_CUDA_TRY(cudaMemsetAsync(W.flag, 0, sizeof(int32_t) * n, s));
    GNN_CUDA_TRY(cudaMemsetAsync(W.counters, 0, sizeof(int32_t) * 4, s));
    k_bfs_start<<<blocks_for(n), 256, 0, s>>>(W.parent, W.cmin, W.base, W.order_di, n, W.pos, W.fill, W.front,
                                              W.counters + 1);
    note_launch();
    int32_t nfront = 0;
    GNN_CUDA_TRY(cudaMemcpyAsync(&nfront, W.counters + 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_CUDA_TRY(cudaStreamSynchronize(s));
    int32_t placed = nfront;
    while (placed < n) {
        GNN_CUDA_TRY(cudaMemsetAsync(W.counters + 2, 0, sizeof(int32_t), s));
        k_bfs_expand<<<blocks_for((int64_t)nfront * 32), 256, 0, s>>>(g->rowptr, g->colidx, W.tp, W.tc, W.front,
                                                                       nfront, W.pos, W.ppos, W.flag, W.cand,
                                                                       W.counters + 2);
        note_launch();
        int32_t nc = 0;
        GNN_CUDA_TRY(cudaMemcpyAsync(&nc, W.counters + 2, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
        GNN_CUDA_TRY(cudaStreamSynchronize(s));
        if (nc == 0) return GNN_ERR_DEVICE_CHECK;  // unreachable nodes would mean a broken component map
        k_level_keys<<<blocks_for(nc), 256, 0, s>>>(W.cand, nc, W.ppos, W.rank, W.key64[0]);
        note_launch();
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, W.key64[0], W.key64[1], W.cand, W.front, nc, 0,
                                                     32 + bn, s));
        note_launch();
        k_seg_heads<<<blocks_for(nc), 256, 0, s>>>(W.front, nc, W.parent, W.cand);
        note_launch();
        GNN_CUDA_TRY(cub::DeviceScan::InclusiveScan(W.temp, tb, W.cand, W.seg, MaxOp(), nc, s));
        note_launch();
        k_level_place<<<blocks_for(nc), 256, 0, s>>>(W.front, nc, W.parent, W.seg, W.fill, W.pos);
        k_level_fill<<<blocks_for(nc), 256, 0, s>>>(W.front, nc, W.parent, W.pos, W.fill);
        note_launch(2);
        nfront = nc;
        placed += nc;
    }
    k_rcm_emit<<<blocks_for(n), 256, 0, s>>>(W.pos, n, perm);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

// CSR^T: per-column counts, the row id of every edge, and a stable sort of
// (column, edge) pairs; the sorted edge ids give the transposed column ids
// (source rows, ascending within a column) and carry the edge values.
struct TransposeWs {
    int32_t *cnt, *rowid, *keys_out, *eid[2];
    void *temp;
    size_t temp_bytes, bytes;
};

TransposeWs transpose_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    TransposeWs W;
    const int64_t m = std::max<int64_t>(g->nnz, 1);
    W.cnt = c.take<int32_t>((size_t)g->n_cols + 1);
    W.rowid = c.take<int32_t>((size_t)m);
    W.keys_out = c.take<int32_t>((size_t)m);
    W.eid[0] = c.take<int32_t>((size_t)m);
    W.eid[1] = c.take<int32_t>((size_t)m);
    size_t t = 0, x = 0;
    cub::DeviceRadixSort::SortPairs(nullptr, x, (const int32_t *)nullptr, (int32_t *)nullptr,
                                    (const int32_t *)nullptr, (int32_t *)nullptr, m);
    t = std::max(t, x);
    cub::DeviceScan::ExclusiveSum(nullptr, x, (const int32_t *)nullptr, (int32_t *)nullptr, g->n_cols + 1);
    t = std::max(t, x);
    W.temp_bytes = t;
    W.temp = c.take<uint8_t>(t);
    W.bytes = c.used;
    return W;
}

// per-column edge counts; a column id outside [0, n_cols) sets the error word
__global__ void k_count_cols_checked(const int32_t *__restrict__ colidx, int64_t nnz, int32_t n_cols,
                                     int32_t *__restrict__ cnt, int32_t *err) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) {
        const int32_t j = colidx[e];
        if ((uint32_t)j >= (uint32_t)n_cols) { set_device_error(err, GNN_ERR_DEVICE_CHECK); continue; }
        atomicAdd(&cnt[j], 1);
    }
}

__global__ void k_iota_i64(int32_t *__restrict__ v, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) v[i] = (int32_t)i;
}

__global__ void k_transpose_fill(const int32_t *__restrict__ eid, const int32_t *__restrict__ rowid,
                                 const float *__restrict__ vals, int64_t m, int32_t *__restrict__ colidx_t,
                                 float *__restrict__ vals_t) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < m; k += stride) {
        const int32_t e = eid[k];
        colidx_t[k] = rowid[e];
        if (vals_t) vals_t[k] = vals[e];
    }
}

}  // namespace

size_t transpose_workspace_bytes(const gnn_csr *g) { return transpose_layout(g, nullptr).bytes; }
size_t reorder_workspace_bytes(const gnn_csr *g) { return reorder_layout(g, nullptr).bytes; }
size_t apply_perm_workspace_bytes(const gnn_csr *g) { return perm_layout(g, nullptr).bytes; }

}  // namespace gnn

using namespace gnn;

extern "C" {

gnn_status gnn_reorder_perm(const gnn_csr *g, int32_t kind, uint64_t seed, int32_t *perm, int32_t *inv,
                            void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols) return GNN_ERR_UNSUPPORTED;
    if (kind < GNN_PERM_IDENTITY || kind > GNN_PERM_RCM) return GNN_ERR_INVALID_ARG;
    const int32_t n = g->n_rows;
    if (n == 0) return GNN_OK;
    if (!perm && !inv) return GNN_ERR_INVALID_ARG;
    ReorderWs W = reorder_layout(g, ws);
    if (!ws || ws_bytes < W.bytes) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    int32_t *P = perm ? perm : W.id[1];
    size_t tb = W.temp_bytes;
    if (kind == GNN_PERM_IDENTITY) {
        k_iota<<<blocks_for(n), 256, 0, s>>>(P, n);
        note_launch();
    } else if (kind == GNN_PERM_RANDOM) {
        k_random_keys<<<blocks_for(n), 256, 0, s>>>(W.key64[0], W.id[0], n, seed);
        note_launch();
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, W.key64[0], W.key64[1], W.id[0], P, n, 0, 64, s));
        note_launch();
    } else if (kind == GNN_PERM_DEGREE) {
        GNN_CUDA_TRY(cudaMemsetAsync(W.dout, 0, sizeof(int32_t) * n, s));
        if (g->nnz > 0) {
            k_count_cols<<<std::min(blocks_for(g->nnz), sm_count() * 8), 256, 0, s>>>(g->colidx, g->nnz, W.dout);
            note_launch();
        }
        k_degree_keys<<<blocks_for(n), 256, 0, s>>>(g->rowptr, W.dout, W.key32[0], W.id[0], n);
        note_launch();
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, W.key32[0], W.key32[1], W.id[0], P, n, 0, 32, s));
        note_launch();
    } else {
        st = rcm_order(g, W, P, s);
        if (st != GNN_OK) return st;
    }
    if (inv) {
        k_inv_from_perm<<<blocks_for(n), 256, 0, s>>>(P, inv, n);
        note_launch();
    }
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_apply_perm(const gnn_csr *g, const int32_t *perm, const int32_t *inv, int32_t *rowptr_out,
                          int32_t *colidx_out, const void *X, int32_t x_dtype, int32_t F, void *X_out, void *ws,
                          size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols) return GNN_ERR_UNSUPPORTED;
    const int32_t n = g->n_rows;
    const int64_t m = g->nnz;
    if (!perm || !rowptr_out || (m > 0 && !colidx_out)) return GNN_ERR_INVALID_ARG;
    if (X) {
        if (!X_out || (x_dtype != GNN_F32 && x_dtype != GNN_BF16) || F <= 0) return GNN_ERR_INVALID_ARG;
        if (((int64_t)F * (x_dtype == GNN_F32 ? 4 : 2)) % 16 || !aligned16(X) || !aligned16(X_out))
            return GNN_ERR_INVALID_ARG;
    }
    PermWs W = perm_layout(g, ws);
    if (!ws || ws_bytes < W.bytes) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    size_t tb = W.temp_bytes;
    if (n == 0) {
        GNN_CUDA_TRY(cudaMemsetAsync(rowptr_out, 0, sizeof(int32_t), s));
        return GNN_OK;
    }
    const int32_t *I = inv;
    if (!I) {
        k_inv_from_perm<<<blocks_for(n), 256, 0, s>>>(perm, W.inv, n);
        note_launch();
        I = W.inv;
    }
    k_new_degrees<<<blocks_for(n + 1), 256, 0, s>>>(g->rowptr, perm, n, W.deg);
    note_launch();
    GNN_CUDA_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.deg, rowptr_out, n + 1, s));
    note_launch();
    if (m > 0) {
        k_relabel_keys<<<blocks_for((int64_t)n * 32), 256, 0, s>>>(g->rowptr, g->colidx, perm, I, rowptr_out, n,
                                                                   W.key[0]);
        note_launch();
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortKeys(W.temp, tb, W.key[0], W.key[1], m, 0, 32 + bits_for(n), s));
        note_launch();
        k_low_words<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(W.key[1], m, colidx_out);
        note_launch();
    }
    if (X) {
        const int64_t chunks = (int64_t)F * (x_dtype == GNN_F32 ? 4 : 2) / 16;
        k_gather_rows<<<blocks_for((int64_t)n * 32), 256, 0, s>>>(static_cast<const uint4 *>(X), perm, n, chunks,
                                                                   static_cast<uint4 *>(X_out));
        note_launch();
    }
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_csr_transpose(const gnn_csr *g, int32_t *rowptr_t, int32_t *colidx_t, float *values_t, void *ws,
                             size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!rowptr_t || (g->nnz > 0 && !colidx_t)) return GNN_ERR_INVALID_ARG;
    if (values_t && !g->values) return GNN_ERR_INVALID_ARG;
    TransposeWs W = transpose_layout(g, ws);
    if (!ws || ws_bytes < W.bytes) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const int64_t m = g->nnz;
    const int32_t nc = g->n_cols;
    size_t tb = W.temp_bytes;
    GNN_CUDA_TRY(cudaMemsetAsync(W.cnt, 0, sizeof(int32_t) * ((size_t)nc + 1), s));
    if (m > 0) {
        int32_t *err = device_error_word();
        if (!err) return GNN_ERR_CUDA;
        k_count_cols_checked<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(g->colidx, m, nc, W.cnt, err);
        k_edge_rows<<<blocks_for((int64_t)g->n_rows * 32), 256, 0, s>>>(g->rowptr, g->n_rows, W.rowid);
        k_iota_i64<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(W.eid[0], m);
        note_launch(3);
        GNN_CUDA_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, g->colidx, W.keys_out, W.eid[0], W.eid[1], m, 0,
                                                     bits_for(nc), s));
        note_launch();
        k_transpose_fill<<<std::min(blocks_for(m), sm_count() * 8), 256, 0, s>>>(W.eid[1], W.rowid, g->values, m,
                                                                                 colidx_t, values_t);
        note_launch();
    }
    GNN_CUDA_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.cnt, rowptr_t, nc + 1, s));
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

}  // extern "C"
