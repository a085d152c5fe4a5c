// Workspace sizing for every operation, and entry points whose kernels live
// in later translation units of this library.
#include "common.cuh"

namespace gnn {
size_t agg_workspace_bytes(const gnn_csr *g, int32_t op, int32_t x_dtype, int32_t F);
size_t gatv2_workspace_bytes(const gnn_csr *g, int32_t F_in, int32_t heads, int32_t head_dim,
                             int32_t esize);
size_t gt_tiles_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim);
size_t reorder_workspace_bytes(const gnn_csr *g);
size_t apply_perm_workspace_bytes(const gnn_csr *g);
size_t blocksparse_workspace_bytes(const gnn_csr *g);
size_t tile_spmm_workspace_bytes(const gnn_csr *g, int32_t F);
size_t transpose_workspace_bytes(const gnn_csr *g);
size_t gt_bwd_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim);
size_t gatv2_bwd_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim);
size_t graph_stats_workspace_bytes(const gnn_csr *g);
gnn_status check_csr_args(const gnn_csr *g);
}  // namespace gnn

using namespace gnn;

extern "C" size_t gnn_workspace_size(int32_t op, const gnn_csr *g, int32_t F, int32_t heads,
                                     int32_t head_dim) {
    if (check_csr_args(g) != GNN_OK) return 0;
    const int32_t esize = (op & GNN_OP_FLAG_BF16) ? 2 : 4;
    switch (op & ~GNN_OP_FLAG_BF16) {
        case GNN_OP_SPMM:
        case GNN_OP_SUM:
        case GNN_OP_MEAN:
        case GNN_OP_MAX:
        case GNN_OP_MIN:
            return agg_workspace_bytes(g, op & ~GNN_OP_FLAG_BF16, GNN_F32, F);
        case GNN_OP_GATV2:
            return gatv2_workspace_bytes(g, F, heads, head_dim, esize);
        case GNN_OP_GT:
            return gt_tiles_workspace_bytes(g, heads, head_dim);  // covers the CSR path too
        case GNN_OP_REORDER:
            return reorder_workspace_bytes(g);
        case GNN_OP_APPLY_PERM:
            return apply_perm_workspace_bytes(g);
        case GNN_OP_BLOCKSPARSE:
            return blocksparse_workspace_bytes(g);
        case GNN_OP_SPMM_BLOCKSPARSE:
            return tile_spmm_workspace_bytes(g, F);
        case GNN_OP_TRANSPOSE:
            return transpose_workspace_bytes(g);
        case GNN_OP_GT_BACKWARD:
            return gt_bwd_workspace_bytes(g, heads, head_dim);
        case GNN_OP_GATV2_BACKWARD:
            return gatv2_bwd_workspace_bytes(g, heads, head_dim);
        case GNN_OP_GRAPH_STATS:
            return graph_stats_workspace_bytes(g);
        default:
            return 0;
    }
}
