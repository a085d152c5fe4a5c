// Library runtime: launch counter, device error word, status strings,
// graph preparation (step a0) and CSR validation.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace gnn {

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

gnn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GNN_OK : GNN_ERR_CUDA; }

// One error word per device (the library supports devices 0..63).
static __device__ int32_t d_error_word;

int32_t *device_error_word() {
    static int32_t *ptrs[64] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, d_error_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int32_t *>(p);
    }
    return ptrs[dev];
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

// ------------------------------------------------------------ step a0

// d_out[j] = occurrences of j in colidx (int32 atomics: exact, order-free).
__global__ void k_count_out_degree(const int32_t *__restrict__ colidx, int64_t nnz,
                                   int32_t n_cols, int32_t *__restrict__ d_out,
                                   int32_t *err) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nnz; e += stride) {
        int32_t j = colidx[e];
        if ((uint32_t)j >= (uint32_t)n_cols) { set_device_error(err, GNN_ERR_DEVICE_CHECK); continue; }
        atomicAdd(&d_out[j], 1);
    }
}

// dinv_in[i] = 1/sqrt(d_in(i)) (0 for an empty row); dinv_out likewise.
__global__ void k_inv_sqrt_degrees(const int32_t *__restrict__ rowptr, int32_t n_rows,
                                   const int32_t *__restrict__ d_out, int32_t n_cols,
                                   float *__restrict__ dinv_in, float *__restrict__ dinv_out) {
    int32_t stride = gridDim.x * blockDim.x;
    int32_t n = n_rows > n_cols ? n_rows : n_cols;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        if (i < n_rows) {
            int32_t d = rowptr[i + 1] - rowptr[i];
            dinv_in[i] = d > 0 ? rsqrtf((float)d) : 0.f;
        }
        if (i < n_cols) {
            int32_t d = d_out[i];
            dinv_out[i] = d > 0 ? rsqrtf((float)d) : 0.f;
        }
    }
}

// Structural checks of a CSR; failures set the error word.
__global__ void k_validate_csr(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ colidx,
                               int32_t n_rows, int32_t n_cols, int64_t nnz, int32_t *err) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_rows; i += stride) {
        int32_t b = rowptr[i], e = rowptr[i + 1];
        if ((i == 0 && b != 0) || e < b || (i == n_rows - 1 && (int64_t)e != nnz) || b < 0 ||
            (int64_t)e > nnz) {
            set_device_error(err, GNN_ERR_DEVICE_CHECK);
            continue;
        }
        int32_t prev = -1;
        for (int32_t k = b; k < e; ++k) {
            int32_t j = colidx[k];
            if (j <= prev || j >= n_cols) { set_device_error(err, GNN_ERR_DEVICE_CHECK); break; }
            prev = j;
        }
    }
}

}  // namespace gnn

using namespace gnn;

namespace {
struct PrepLayout {
    int32_t *d_out;
    float *dinv_in;
    float *dinv_out;
    int32_t *run_first_row;  // [n_runs(kRunEdges) + 1]
    size_t bytes;
};

PrepLayout prep_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    PrepLayout L;
    L.d_out = c.take<int32_t>((size_t)g->n_cols);
    L.dinv_in = c.take<float>((size_t)g->n_rows);
    L.dinv_out = c.take<float>((size_t)g->n_cols);
    L.run_first_row = c.take<int32_t>((size_t)n_runs(g->nnz, kRunEdges) + 1);
    L.bytes = c.used;
    return L;
}

// run_first_row[w] = first row r with rowptr[r] >= w * E (w < n_runs), and
// run_first_row[n_runs] = n_rows.
__global__ void k_run_first_row(const int32_t *__restrict__ rowptr, int32_t n_rows, int32_t E,
                                int32_t n_run, int32_t *__restrict__ out) {
    int32_t w = blockIdx.x * blockDim.x + threadIdx.x;
    if (w > n_run) return;
    if (w == n_run) { out[w] = n_rows; return; }
    int32_t e = w * E;
    int32_t lo = 0, hi = n_rows;
    while (lo < hi) {
        int32_t mid = (lo + hi) >> 1;
        if (rowptr[mid] < e) lo = mid + 1; else hi = mid;
    }
    out[w] = lo;
}
}  // namespace

namespace gnn {
// Shared with the other translation units through these accessors.
void prep_pointers(const gnn_csr *g, const void *prep, const int32_t **d_out,
                   const float **dinv_in, const float **dinv_out) {
    PrepLayout L = prep_layout(g, const_cast<void *>(prep));
    *d_out = L.d_out;
    *dinv_in = L.dinv_in;
    *dinv_out = L.dinv_out;
}

const int32_t *prep_run_table(const gnn_csr *g, const void *prep) {
    return prep_layout(g, const_cast<void *>(prep)).run_first_row;
}

gnn_status check_csr_args(const gnn_csr *g) {
    if (!g || !g->rowptr || g->n_rows < 0 || g->n_cols < 0 || g->nnz < 0 ||
        g->nnz >= ((int64_t)1 << 31))
        return GNN_ERR_INVALID_ARG;
    if (g->nnz > 0 && !g->colidx) return GNN_ERR_INVALID_ARG;
    return GNN_OK;
}
}  // namespace gnn

extern "C" {

size_t gnn_graph_prepare_size(const gnn_csr *g) {
    if (check_csr_args(g) != GNN_OK) return 0;
    return prep_layout(g, nullptr).bytes;
}

gnn_status gnn_graph_prepare(const gnn_csr *g, void *prep, size_t prep_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!prep || !aligned256(prep)) return GNN_ERR_INVALID_ARG;
    PrepLayout L = prep_layout(g, prep);
    if (prep_bytes < L.bytes) return GNN_ERR_WORKSPACE;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    if (g->n_cols > 0) {
        cudaError_t e = cudaMemsetAsync(L.d_out, 0, sizeof(int32_t) * (size_t)g->n_cols, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    int sms = sm_count();
    if (g->nnz > 0) {
        int blocks = (int)std::min<int64_t>((g->nnz + 255) / 256, (int64_t)sms * 8);
        k_count_out_degree<<<blocks, 256, 0, s>>>(g->colidx, g->nnz, g->n_cols, L.d_out, err);
        note_launch();
        GNN_LAUNCH_CHECK();
    }
    int32_t n = std::max(g->n_rows, g->n_cols);
    if (n > 0) {
        int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sms * 8);
        k_inv_sqrt_degrees<<<blocks, 256, 0, s>>>(g->rowptr, g->n_rows, L.d_out, g->n_cols,
                                                  L.dinv_in, L.dinv_out);
        note_launch();
        GNN_LAUNCH_CHECK();
    }
    int32_t nr = (int32_t)n_runs(g->nnz, kRunEdges);
    k_run_first_row<<<(nr + 1 + 255) / 256, 256, 0, s>>>(g->rowptr, g->n_rows, kRunEdges, nr,
                                                         L.run_first_row);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_csr_validate(const gnn_csr *g, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    if (g->n_rows == 0) return GNN_OK;
    int blocks = (int)std::min<int64_t>((g->n_rows + 255) / 256, (int64_t)sm_count() * 8);
    k_validate_csr<<<blocks, 256, 0, as_stream(stream)>>>(g->rowptr, g->colidx, g->n_rows,
                                                          g->n_cols, g->nnz, err);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_last_device_error(void *stream, int32_t *code) {
    if (!code) return GNN_ERR_INVALID_ARG;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    *code = v;
    return GNN_OK;
}

const char *gnn_status_string(int32_t s) {
    switch (s) {
        case GNN_OK: return "ok";
        case GNN_ERR_INVALID_ARG: return "invalid argument";
        case GNN_ERR_UNSUPPORTED: return "unsupported";
        case GNN_ERR_WORKSPACE: return "workspace too small";
        case GNN_ERR_CUDA: return "CUDA error";
        case GNN_ERR_DEVICE_CHECK: return "device-side check failed";
        case GNN_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

uint64_t gnn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *gnn_version(void) { return "libgnn 0.1 sm_103a"; }

}  // extern "C"
