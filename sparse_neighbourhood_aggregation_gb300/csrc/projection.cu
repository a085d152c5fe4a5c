// Step a3: dense projection C = H W on the tcgen05 tensor cores (bf16).
#include "common.cuh"

namespace gnn {

gnn_status projection_tc(const void *, int64_t, int32_t, const void *, int32_t, void *, cudaStream_t) {
    return GNN_ERR_UNSUPPORTED;
}

}  // namespace gnn
