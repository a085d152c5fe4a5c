// Library runtime: launch counter, device error word, status strings,
// graph preparation (step a0) and CSR validation.
#include <atomic>
#include <mutex>

#include <cub/device/device_scan.cuh>

#include <set>
#include <tuple>
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

cudaError_t func_attr(const void *fn, cudaFuncAttribute attr, int value) {
    static std::mutex mu;
    static std::set<std::tuple<const void *, int, int, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(fn, dev, (int)attr, value);
    std::lock_guard<std::mutex> lk(mu);
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, attr, value);
    if (e == cudaSuccess) done.insert(key);
    return e;
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

// Row-end bits of the edge list: bit (e & 31) of word e >> 5 is set when
// edge e is the last edge of its row.  Rows are independent, so the ORs
// commute and the result is exact.
__global__ void k_row_end_flags(const int32_t *__restrict__ rowptr, int32_t n_rows, int64_t nnz,
                                uint32_t *__restrict__ flags, int32_t *err) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
        int32_t b = rowptr[r], e = rowptr[r + 1];
        if (e <= b) continue;
        if (b < 0 || (int64_t)e > nnz) { set_device_error(err, GNN_ERR_DEVICE_CHECK); continue; }
        atomicOr(flags + ((e - 1) >> 5), 1u << ((e - 1) & 31));
    }
}

__global__ void k_popc_words(const uint32_t *__restrict__ flags, int32_t n, int32_t *__restrict__ cnt) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) cnt[i] = __popc(flags[i]);
}

// ne_rows[k] = the k-th non-empty row: its rank is the number of row ends
// before its own last edge, read from the scanned window counts.
__global__ void k_nonempty_rows(const int32_t *__restrict__ rowptr, int32_t n_rows, int64_t nnz,
                                const uint32_t *__restrict__ flags,
                                const int32_t *__restrict__ win_rowbase,
                                int32_t *__restrict__ ne_rows) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
        int32_t b = rowptr[r], e = rowptr[r + 1];
        if (e <= b || b < 0 || (int64_t)e > nnz) continue;
        int32_t last = e - 1;
        int32_t k = win_rowbase[last >> 5] + __popc(flags[last >> 5] & ((1u << (last & 31)) - 1u));
        if ((uint32_t)k < (uint32_t)n_rows) ne_rows[k] = r;
    }
}

// win_rowstart[win] = first edge of the row holding edge 32*win.
__global__ void k_win_rowstart(const int32_t *__restrict__ rowptr, int32_t n_rows, int32_t n_win,
                               const int32_t *__restrict__ win_rowbase,
                               const int32_t *__restrict__ ne_rows, int32_t *__restrict__ out) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_win; i += stride) {
        const int32_t k = win_rowbase[i];
        const int32_t r = (uint32_t)k < (uint32_t)n_rows ? ne_rows[k] : 0;
        out[i] = rowptr[r];
    }
}

// sp_begin[w] = first edge of span w.  The nominal span is [w*S, (w+1)*S);
// a row of degree <= S that crosses w*S belongs whole to span w-1, so span w
// starts after it; a heavier row is cut at w*S.  sp_begin[n_spans] = nnz.
__global__ void k_span_begin(const int32_t *__restrict__ rowptr, int64_t nnz, int32_t n_spans, int32_t es,
                             const uint32_t *__restrict__ flags,
                             const int32_t *__restrict__ win_rowbase,
                             const int32_t *__restrict__ ne_rows, int32_t n_rows,
                             int32_t *__restrict__ out) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t w = blockIdx.x * blockDim.x + threadIdx.x; w <= n_spans; w += stride) {
        if (w == n_spans) { out[w] = (int32_t)nnz; continue; }
        const int32_t e = w << es;
        if (e == 0 || ((flags[(e - 1) >> 5] >> ((e - 1) & 31)) & 1u)) { out[w] = e; continue; }
        const int32_t k = win_rowbase[e >> 5];
        const int32_t r = (uint32_t)k < (uint32_t)n_rows ? ne_rows[k] : 0;
        const int32_t s = rowptr[r], t = rowptr[r + 1];
        out[w] = (t - s > (1 << es)) ? e : t;
    }
}

// Work items of the heavy-row finalising kernel: a row of degree > S touches
// spans s0..s1 and leaves one piece in each; its pieces are taken kFixChunk
// at a time, item {row, rowptr[row], rowptr[row+1], chunk index}.  A row's
// items are contiguous (one atomic reservation); rows come in any order.
// items_count holds their number.
__global__ void k_heavy_items(const int32_t *__restrict__ rowptr, int32_t n_rows, int32_t es, int64_t cap,
                              int4 *__restrict__ items, int32_t *__restrict__ items_count,
                              int32_t *err) {
    int32_t stride = gridDim.x * blockDim.x;
    for (int32_t r = blockIdx.x * blockDim.x + threadIdx.x; r < n_rows; r += stride) {
        const int32_t rb = rowptr[r], re = rowptr[r + 1];
        if (re - rb <= (1 << es)) continue;
        const int32_t np = ((re - 1) >> es) - (rb >> es) + 1;
        const int32_t nch = (np + kFixChunk - 1) / kFixChunk;
        const int32_t base = atomicAdd(items_count, nch);
        if ((int64_t)base + nch > cap) { set_device_error(err, GNN_ERR_DEVICE_CHECK); continue; }
        for (int32_t c = 0; c < nch; ++c) items[base + c] = make_int4(r, rb, re, c);
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
    uint32_t *win_flags;     // [n_win] row-end bits per 32-edge window
    int32_t *win_count;      // [n_win] popcounts (scan input)
    int32_t *win_rowbase;    // [n_win] rank among non-empty rows of the row holding edge 32*win
    int32_t *ne_rows;        // [n_rows] non-empty rows, ascending (first n_nonempty entries)
    int32_t *sp_begin;       // [n_spans + 1] first edge of each edge span
    int32_t *win_rowstart;   // [n_win] first edge of the row holding edge 32*win
    int4 *items;             // [span_item_cap(nnz)] heavy-row chunks for the finalising kernel
    int32_t *items_count;    // [1]
    int32_t n_spans;
    void *scan_tmp;
    size_t scan_tmp_bytes;
    int32_t n_win;
    size_t bytes;
};

PrepLayout prep_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    PrepLayout L;
    L.d_out = c.take<int32_t>((size_t)g->n_cols);
    L.dinv_in = c.take<float>((size_t)g->n_rows);
    L.dinv_out = c.take<float>((size_t)g->n_cols);
    L.run_first_row = c.take<int32_t>((size_t)n_runs(g->nnz, kRunEdges) + 1);
    L.n_win = (int32_t)((g->nnz + 31) / 32);
    L.win_flags = c.take<uint32_t>((size_t)L.n_win);
    L.win_count = c.take<int32_t>((size_t)L.n_win);
    L.win_rowbase = c.take<int32_t>((size_t)L.n_win);
    L.ne_rows = c.take<int32_t>((size_t)g->n_rows);
    L.n_spans = (int32_t)n_spans_of(g->nnz);
    L.sp_begin = c.take<int32_t>((size_t)L.n_spans + 1);
    L.win_rowstart = c.take<int32_t>((size_t)L.n_win);
    L.items = c.take<int4>((size_t)span_item_cap(g->nnz));
    L.items_count = c.take<int32_t>(1);
    L.scan_tmp_bytes = 0;
    if (L.n_win > 0)
        cub::DeviceScan::ExclusiveSum(nullptr, L.scan_tmp_bytes, (const int32_t *)nullptr,
                                      (int32_t *)nullptr, L.n_win);
    L.scan_tmp = c.take<uint8_t>(L.scan_tmp_bytes);
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

void prep_span_tables(const gnn_csr *g, const void *prep, const uint32_t **win_flags,
                      const int32_t **win_rowbase, const int32_t **ne_rows,
                      const int32_t **sp_begin, const int4 **items,
                      const int32_t **items_count, const int32_t **win_rowstart) {
    PrepLayout L = prep_layout(g, const_cast<void *>(prep));
    *win_rowstart = L.win_rowstart;
    *sp_begin = L.sp_begin;
    *items = L.items;
    *items_count = L.items_count;
    *win_flags = L.win_flags;
    *win_rowbase = L.win_rowbase;
    *ne_rows = L.ne_rows;
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
    // edge-span tables: row-end bits, their window ranks and the non-empty rows
    if (L.n_win > 0 && g->n_rows > 0) {
        cudaError_t e = cudaMemsetAsync(L.win_flags, 0, sizeof(uint32_t) * (size_t)L.n_win, s);
        if (e != cudaSuccess) return cuda_status(e);
        // ranks past the last non-empty row read row 0, a valid index
        e = cudaMemsetAsync(L.ne_rows, 0, sizeof(int32_t) * (size_t)g->n_rows, s);
        if (e != cudaSuccess) return cuda_status(e);
        int rb = (int)std::min<int64_t>((g->n_rows + 255) / 256, (int64_t)sms * 8);
        int wb = (int)std::min<int64_t>((L.n_win + 255) / 256, (int64_t)sms * 8);
        k_row_end_flags<<<rb, 256, 0, s>>>(g->rowptr, g->n_rows, g->nnz, L.win_flags, err);
        k_popc_words<<<wb, 256, 0, s>>>(L.win_flags, L.n_win, L.win_count);
        note_launch(2);
        GNN_LAUNCH_CHECK();
        size_t tb = L.scan_tmp_bytes;
        e = cub::DeviceScan::ExclusiveSum(L.scan_tmp, tb, L.win_count, L.win_rowbase, L.n_win, s);
        if (e != cudaSuccess) return cuda_status(e);
        k_nonempty_rows<<<rb, 256, 0, s>>>(g->rowptr, g->n_rows, g->nnz, L.win_flags,
                                           L.win_rowbase, L.ne_rows);
        k_win_rowstart<<<wb, 256, 0, s>>>(g->rowptr, g->n_rows, L.n_win, L.win_rowbase, L.ne_rows,
                                          L.win_rowstart);
        note_launch();
        const int sb = (int)std::min<int64_t>((L.n_spans + 1 + 255) / 256, (int64_t)sms * 8);
        k_span_begin<<<sb, 256, 0, s>>>(g->rowptr, g->nnz, L.n_spans, span_shift(g->nnz), L.win_flags,
                                        L.win_rowbase,
                                        L.ne_rows, g->n_rows, L.sp_begin);
        e = cudaMemsetAsync(L.items_count, 0, sizeof(int32_t), s);
        if (e != cudaSuccess) return cuda_status(e);
        k_heavy_items<<<rb, 256, 0, s>>>(g->rowptr, g->n_rows, span_shift(g->nnz), span_item_cap(g->nnz),
                                         L.items,
                                         L.items_count, err);
        note_launch(3);
        GNN_LAUNCH_CHECK();
    }
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
