// Adaptive choice of backend from graph statistics.
//
// IO-aware GNN layers, Section 5 (an adaptive runtime that picks between the
// CSR kernels and the block-sparse tensor-core path from the degree skew,
// the local density and the feature size) and Appendix B.1 (Table 5: the
// degree skewness of each graph).  gnn_graph_stats_compute measures the
// statistics on the GPU: the moments of the row lengths in one pass (fixed
// per-block order, then the blocks summed on the host in order, so the
// result is deterministic) and the local density from the block-sparse plan
// at fill 0 (edges per listed 128 x 16 column block).  gnn_select_backend is
// a pure host rule on those statistics.
//
// The rule's break-even densities are measured on GB300 on the clustered
// 262K-node graph (20.3M edges, 46,240 listed blocks, 439 edges a block):
// GCN SpMM of bf16 [N, 256] features took 0.909 ms on the CSR edge spans and
// 0.327 ms on tcgen05 tiles, i.e. 22.3 G edges/s against 141 M blocks/s, so
// the tiles win above 158 edges per block; GT attention (8 heads x 32) took
// 2.11 ms on CSR and 0.621 ms on tiles, 9.6 G edges/s against 74.5 M
// blocks/s, break-even 129 edges per block.  Both rates scale with the
// feature width alike, so the break-even does not depend on F.  The CSR
// kernels are degree-aware by construction (edge spans and runs cut heavy
// rows whatever the skew), so the skew selects nothing there; it is reported.
#include <cmath>
#include <vector>

#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);
size_t blocksparse_workspace_bytes(const gnn_csr *g);

namespace {

constexpr int kMomBlocks = 256;
constexpr int kMomThreads = 256;
constexpr double kSpmmTileEdgesPerBlock = 158.0;
constexpr double kGtTileEdgesPerBlock = 129.0;

struct Moments {
    long long s1, s2;  // sum d, sum d^2 (exact: sum d^2 <= max d * nnz < 2^62)
    double s3;         // sum d^3
    long long mx;
};

// Per-block sums of d, d^2, d^3 and max d over the row lengths (grid-stride
// rows, then a fixed-order tree in shared memory).
__global__ void __launch_bounds__(kMomThreads) k_degree_moments(const int32_t *__restrict__ rowptr, int32_t n,
                                                                Moments *__restrict__ part) {
    long long s1 = 0, s2 = 0, mx = 0;
    double s3 = 0.0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const long long d = (long long)__ldg(rowptr + i + 1) - __ldg(rowptr + i);
        s1 += d;
        s2 += d * d;
        s3 += (double)d * (double)d * (double)d;
        mx = d > mx ? d : mx;
    }
    __shared__ Moments sh[kMomThreads];
    sh[threadIdx.x] = Moments{s1, s2, s3, mx};
    __syncthreads();
    for (int o = kMomThreads / 2; o > 0; o >>= 1) {
        if ((int)threadIdx.x < o) {
            Moments &a = sh[threadIdx.x];
            const Moments &b = sh[threadIdx.x + o];
            a.s1 += b.s1;
            a.s2 += b.s2;
            a.s3 += b.s3;
            a.mx = b.mx > a.mx ? b.mx : a.mx;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) part[blockIdx.x] = sh[0];
}

}  // namespace

size_t graph_stats_workspace_bytes(const gnn_csr *g) {
    return round_up(sizeof(Moments) * kMomBlocks, 256) + blocksparse_workspace_bytes(g);
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_graph_stats_compute(const gnn_csr *g, gnn_graph_stats *out, void *ws, size_t ws_bytes,
                                              void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!out) return GNN_ERR_INVALID_ARG;
    *out = gnn_graph_stats{};
    out->n_rows = g->n_rows;
    out->nnz = g->nnz;
    if (g->n_rows == 0) return GNN_OK;
    if (!ws || ws_bytes < graph_stats_workspace_bytes(g)) return GNN_ERR_WORKSPACE;
    cudaStream_t s = as_stream(stream);
    Moments *part = static_cast<Moments *>(ws);
    const size_t part_bytes = round_up(sizeof(Moments) * kMomBlocks, 256);
    k_degree_moments<<<kMomBlocks, kMomThreads, 0, s>>>(g->rowptr, g->n_rows, part);
    note_launch();
    GNN_LAUNCH_CHECK();
    std::vector<Moments> h(kMomBlocks);
    if (cudaMemcpyAsync(h.data(), part, sizeof(Moments) * kMomBlocks, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return GNN_ERR_CUDA;
    long long s1 = 0, s2 = 0, mx = 0;
    double s3 = 0.0;
    for (const Moments &m : h) {
        s1 += m.s1;
        s2 += m.s2;
        s3 += m.s3;
        mx = m.mx > mx ? m.mx : mx;
    }
    const double n = (double)g->n_rows;
    const double mean = (double)s1 / n;
    const double e2 = (double)s2 / n, e3 = s3 / n;
    double m2 = e2 - mean * mean;
    if (m2 < 0.0) m2 = 0.0;
    const double m3 = e3 - 3.0 * mean * e2 + 2.0 * mean * mean * mean;
    out->max_degree = (int32_t)mx;
    out->mean_degree = mean;
    out->degree_std = sqrt(m2);
    out->degree_skewness = m2 > 0.0 ? m3 / (m2 * sqrt(m2)) : 0.0;
    // local density: listed 128 x 16 blocks of the block-sparse plan at fill 0
    gnn_blocksparse bs{};
    size_t bytes = 0;
    st = gnn_blocksparse_plan(g, 0.f, static_cast<char *>(ws) + part_bytes, ws_bytes - part_bytes, &bs, &bytes,
                              stream);
    if (st != GNN_OK) return st;
    out->n_blocks = bs.n_blocks;
    out->edges_per_block = bs.n_blocks > 0 ? (double)g->nnz / (double)bs.n_blocks : 0.0;
    return GNN_OK;
}

extern "C" int32_t gnn_select_backend(const gnn_graph_stats *s, int32_t op, int32_t dtype, int32_t F, int32_t heads,
                                      int32_t head_dim, float *fill_threshold) {
    if (fill_threshold) *fill_threshold = 0.f;
    if (!s || s->nnz == 0 || dtype != GNN_BF16) return GNN_BACKEND_CSR;
    if (op == GNN_OP_SPMM) {
        if (F <= 0 || F % 64) return GNN_BACKEND_CSR;
        return s->edges_per_block >= kSpmmTileEdgesPerBlock ? GNN_BACKEND_TILES : GNN_BACKEND_CSR;
    }
    if (op == GNN_OP_GT) {
        if (heads <= 0 || (head_dim != 32 && head_dim != 64)) return GNN_BACKEND_CSR;
        return s->edges_per_block >= kGtTileEdgesPerBlock ? GNN_BACKEND_TILES : GNN_BACKEND_CSR;
    }
    return GNN_BACKEND_CSR;
}
