// Entry points declared in gnn.h whose kernels are not built yet: each
// returns GNN_ERR_UNSUPPORTED without launching anything.
#include "common.cuh"

namespace gnn {
size_t blocksparse_workspace_bytes(const gnn_csr *) { return 0; }

gnn_status gt_attn_tiles(const gnn_csr *, const gnn_blocksparse *, const void *, const void *,
                         const void *, int32_t, int32_t, float, float *, float *, void *, size_t,
                         cudaStream_t) {
    return GNN_ERR_UNSUPPORTED;
}
}  // namespace gnn

extern "C" {

gnn_status gnn_blocksparse_plan(const gnn_csr *, float, void *, size_t, gnn_blocksparse *,
                                size_t *, void *) {
    return GNN_ERR_UNSUPPORTED;
}

gnn_status gnn_blocksparse_build(const gnn_csr *, gnn_blocksparse *, void *, size_t, void *,
                                 size_t, void *) {
    return GNN_ERR_UNSUPPORTED;
}

}  // extern "C"
