// Entry points declared in gnn.h whose kernels are not built yet: each
// returns GNN_ERR_UNSUPPORTED without launching anything.
#include "common.cuh"

namespace gnn {

gnn_status gt_attn_tiles(const gnn_csr *, const gnn_blocksparse *, const void *, const void *,
                         const void *, int32_t, int32_t, float, float *, float *, void *, size_t,
                         cudaStream_t) {
    return GNN_ERR_UNSUPPORTED;
}
}  // namespace gnn

extern "C" {

}  // extern "C"
