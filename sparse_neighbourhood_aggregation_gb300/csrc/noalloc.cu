// Segment sum for callers that cannot allocate device memory: the scratch
// space gnn_segment_reduce_sum takes from the caller's workspace comes from
// a fixed, library-owned device array instead.
#include <mutex>

#include "common.cuh"

namespace gnn {
gnn_status check_agg_args(const gnn_csr *g, const void *prep, int32_t norm, const void *X,
                          int32_t x_dtype, int32_t F, const float *Y, const int32_t *argmax,
                          int32_t mapping);
}

namespace {

// Scratch of gnn_segment_reduce_sum_noalloc.  One copy per device, held for
// the life of the process.  In host code this name is only a host-side
// stand-in for the symbol, never a device address: the kernel gets the
// address that cudaGetSymbolAddress returns for the current device.
__device__ __align__(256) unsigned char g_noalloc_scratch[GNN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up on
// the first call per device and cached; nullptr if the lookup fails.  The
// cache is keyed by device ordinal, so it does not survive cudaDeviceReset
// (the module, and with it the array, may be reloaded elsewhere).
void *noalloc_scratch_address() {
    static void *addr[kMaxDevices] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" gnn_status gnn_segment_reduce_sum_noalloc(const gnn_csr *g, const void *prep,
                                                     const void *X, int32_t x_dtype, int32_t F,
                                                     float *Y, void *stream) {
    // the checks of gnn_segment_reduce_sum, with the same codes, before the
    // scratch is touched: a rejected call launches nothing
    const gnn_status st = gnn::check_agg_args(g, prep, GNN_NORM_NONE, X, x_dtype, F, Y, nullptr,
                                              GNN_MAP_AUTO);
    if (st != GNN_OK) return st;
    if (g->n_rows == 0) return GNN_OK;
    const size_t need = gnn_workspace_size(GNN_OP_SUM, g, F, 0, 0);
    if (need > GNN_NOALLOC_SCRATCH_BYTES) return GNN_ERR_WORKSPACE;
    void *ws = noalloc_scratch_address();
    if (!ws) return GNN_ERR_CUDA;
    // the kernel expects its partial sums and counters to start at zero
    if (need > 0) {
        cudaError_t e = cudaMemsetAsync(ws, 0, need, gnn::as_stream(stream));
        if (e != cudaSuccess) return gnn::cuda_status(e);
    }
    return gnn_segment_reduce_sum(g, prep, X, x_dtype, F, Y, ws, need, stream);
}
