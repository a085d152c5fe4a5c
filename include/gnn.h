/*
 * gnn.h -- C ABI of libgnn, CSR neighbourhood aggregation for GNN layers on
 * one NVIDIA GB300 (sm_103a).
 *
 * The operations follow "On efficient scaling of GNNs via IO-aware layer
 * implementations" (cited as "IO-aware GNN layers"): SpMM convolutions
 * (Section 2.2 (i), Appendix D.4), degree-aware segment reductions
 * (Section 2.2 (ii), Appendix D.1) and fused CSR attention for GATv2 and the
 * Graph Transformer (Section 2.2 (iii), Section 3.2, Appendix D.2), plus the
 * 16x16 block-sparse tensor-core layout (Section 3.3, Appendix D.3) and
 * vertex reordering (Section 4.1; RCM as in "A High-Throughput Solver for
 * Marginalized Graph Kernels on GPU", graph reordering section).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Graph: CSR by destination.  Row i lists the source nodes j of the edges
 *   j -> i in colidx[rowptr[i] .. rowptr[i+1]), ascending and without
 *   duplicates; N(i) includes i only if the graph stores a self-loop (the
 *   library never adds one).  Indices are int32 (nnz < 2^31).
 * Memory: every array argument is a DEVICE pointer owned by the caller unless
 *   the comment says "host".  The library never allocates device memory;
 *   scratch space comes from the caller through (ws, ws_bytes), sized by
 *   gnn_workspace_size().  A workspace must be zero-filled before its first
 *   use; every call leaves the parts that the next call of the same
 *   operation on the same graph and feature width needs at zero, so
 *   repeated calls need no further cudaMemset.  Other parts keep scratch
 *   (projected rows, partial sums): a buffer moved to another operation,
 *   graph or width needs a fresh zero-fill.  Calls that may overlap on the
 *   GPU need separate workspaces.
 * Features: dense row-major [rows, F].  Rows must start on 16-byte
 *   boundaries: F % 4 == 0 for fp32, F % 8 == 0 for bf16, and every feature
 *   pointer 16-byte aligned.
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Calls are asynchronous on it unless the comment says "synchronous".
 * Errors: arguments are validated on the host before any launch; a failed
 *   check returns GNN_ERR_INVALID_ARG / GNN_ERR_UNSUPPORTED /
 *   GNN_ERR_WORKSPACE and launches nothing.  Launch failures return
 *   GNN_ERR_CUDA.  Device-side checks (gnn_csr_validate, bounded waits) never
 *   trap: they record a code in a device error word, read with
 *   gnn_last_device_error().
 */
#ifndef GNN_H
#define GNN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GNN_OK = 0,
    GNN_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    GNN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype, width) */
    GNN_ERR_WORKSPACE = 3,     /* ws too small */
    GNN_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    GNN_ERR_DEVICE_CHECK = 5,  /* a device-side check failed (see error word) */
    GNN_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out */
} gnn_status;

typedef enum { GNN_F32 = 0, GNN_BF16 = 1 } gnn_dtype;

/* SpMM normalisation (IO-aware GNN layers, Appendix D.4: none/left/right/
 * both).  Edge weight w_ij = v_ij * f, v_ij = values[e] (or 1 if values is
 * NULL), f = 1 (NONE), 1/d_in(i) (LEFT), 1/d_out(j) (RIGHT),
 * 1/sqrt(d_in(i) d_out(j)) (BOTH, the GCN normalisation of Section 2.2 (i)).
 * d_in(i) = row length, d_out(j) = occurrences of j in colidx. */
typedef enum { GNN_NORM_NONE = 0, GNN_NORM_LEFT = 1, GNN_NORM_RIGHT = 2, GNN_NORM_BOTH = 3 } gnn_norm;

/* Kernel mappings (IO-aware GNN layers, Section 4.1 and Appendix E.1, the
 * "dot-aggr" study; Appendix D.1 degree-aware split):
 *   AUTO  -- degree-aware: the edge list is cut into equal runs of edges, one
 *            per warp; short rows are packed several to a warp, rows longer
 *            than a run are split across warps and their partial results
 *            merged (two-phase, deterministic).  Feature-parallel lanes.
 *   FEAT  -- one warp per destination row, lanes over features (coalesced
 *            loads), neighbours visited sequentially.
 *   NEIGH -- one warp per destination row, lanes over neighbours (gather),
 *            a warp reduction per 16-byte feature slice. */
typedef enum { GNN_MAP_AUTO = 0, GNN_MAP_FEAT = 1, GNN_MAP_NEIGH = 2 } gnn_mapping;

typedef struct {
    int32_t n_rows;        /* destination nodes */
    int32_t n_cols;        /* source nodes (== n_rows for a square graph) */
    int64_t nnz;           /* edges = rowptr[n_rows] */
    const int32_t *rowptr; /* device [n_rows+1], rowptr[0] = 0, non-decreasing */
    const int32_t *colidx; /* device [nnz], each in [0, n_cols) */
    const float *values;   /* device [nnz] edge values, or NULL */
} gnn_csr;

/* ---------------------------------------------------------------- prep */

/* Bytes of the prepared-graph buffer for g (host call, no GPU work). */
size_t gnn_graph_prepare_size(const gnn_csr *g);

/* Step a0: per-graph preparation, done once and reused by every call on the
 * same graph (IO-aware GNN layers, Appendix D.4, "normalisation as a
 * preprocessing step" and the graph-structure cache).  Fills `prep` with
 * d_out[n_cols] (int32), 1/sqrt(d_in)[n_rows] and 1/sqrt(d_out)[n_cols]
 * (fp32), and the schedule tables of the aggregation and attention kernels:
 * the first row of every 64-edge run; one row-end bit per edge (a 32-bit
 * word per 32 edges) with, per word, the rank among non-empty rows of the
 * row holding its first edge and that row's first edge; the non-empty rows
 * in order; the first edge of every 64-edge span once a row of degree <= 64
 * is kept whole in the span it starts in; and the rows of degree > 64.
 * prep: device buffer of gnn_graph_prepare_size(g) bytes, 256-byte
 * aligned, owned by the caller.  Asynchronous. */
gnn_status gnn_graph_prepare(const gnn_csr *g, void *prep, size_t prep_bytes, void *stream);

/* Device-side structural check of g: rowptr[0] == 0, non-decreasing,
 * rowptr[n_rows] == nnz, colidx in [0, n_cols), strictly ascending within a
 * row.  A violation sets the device error word to GNN_ERR_DEVICE_CHECK (no
 * trap).  Asynchronous; read the result with gnn_last_device_error. */
gnn_status gnn_csr_validate(const gnn_csr *g, void *stream);

/* Synchronous: waits for `stream`, returns the device error word (GNN_OK if
 * clear) in *code and clears it. */
gnn_status gnn_last_device_error(void *stream, int32_t *code);

/* Operation ids for gnn_workspace_size. */
typedef enum {
    GNN_OP_SPMM = 0, GNN_OP_SUM = 1, GNN_OP_MEAN = 2, GNN_OP_MAX = 3,
    GNN_OP_GATV2 = 4, GNN_OP_GT = 5, GNN_OP_REORDER = 6, GNN_OP_APPLY_PERM = 7,
    GNN_OP_BLOCKSPARSE = 8, GNN_OP_MIN = 9, GNN_OP_SPMM_BLOCKSPARSE = 10, GNN_OP_TRANSPOSE = 11,
    GNN_OP_GT_BACKWARD = 12, GNN_OP_GATV2_BACKWARD = 13, GNN_OP_GRAPH_STATS = 14
} gnn_op;

/* OR-ed into `op` of gnn_workspace_size: size the workspace for bf16 inputs
 * (the attention ops keep their projected features in the input dtype);
 * without it attention workspaces are sized for fp32 inputs. */
#define GNN_OP_FLAG_BF16 0x100

/* Workspace bytes needed by operation `op` on g with feature width F (or
 * heads x head_dim for attention; F is then F_in for GATv2).  Host call. */
size_t gnn_workspace_size(int32_t op, const gnn_csr *g, int32_t F, int32_t heads,
                          int32_t head_dim);

/* ------------------------------------------------------- step a1: SpMM */

/* Y = A_w X  (IO-aware GNN layers, Section 2.2 (i); GCN with
 * norm = GNN_NORM_BOTH).  X [n_cols, F] (fp32 or bf16), Y [n_rows, F] fp32,
 * accumulation fp32.  prep from gnn_graph_prepare (required for LEFT/RIGHT/
 * BOTH, may be NULL for NONE).  mapping: gnn_mapping.  Supported F: fp32
 * 32..1024 and bf16 64..2048 with F / (16 bytes) a power of two. */
gnn_status gnn_spmm(const gnn_csr *g, const void *prep, int32_t norm, const void *X,
                    int32_t x_dtype, int32_t F, float *Y, int32_t mapping, void *ws,
                    size_t ws_bytes, void *stream);

/* ---------------------------------------- step a2: segment reductions */

/* Y[i,:] = sum over j in N(i) of X[j,:]  (IO-aware GNN layers, Section
 * 2.2 (ii)).  Empty rows give 0.  Shapes and F as gnn_spmm.  prep may be
 * NULL; when given, rows of 32 16-byte chunks (fp32 F = 128, bf16 F = 256)
 * run on the edge-span schedule it holds (two launches: the edge stream,
 * then the rows of degree > 64), and other widths use its edge-run table
 * instead of a per-run search. */
gnn_status gnn_segment_reduce_sum(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, void *ws,
                                  size_t ws_bytes, void *stream);

/* Segment sum without a caller workspace.  The paper has no counterpart to
 * this entry point; it exists for callers that cannot allocate device
 * memory themselves: a plugin inside a host framework that owns every device
 * allocation and hands the plugin only its input and output buffers, or a
 * latency-critical loop that must not pay for cudaMalloc's implicit device
 * synchronisation.
 *
 * Computes exactly what gnn_segment_reduce_sum computes, through the same
 * kernel, but its scratch space (heavy-row partial sums and their arrival
 * counters) is a fixed library-owned device array of
 * GNN_NOALLOC_SCRATCH_BYTES bytes.  Every GPU that loads the library holds
 * that array until the process exits.  The call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * Size limit: the problem must satisfy
 *   gnn_workspace_size(GNN_OP_SUM, g, F, 0, 0) <= GNN_NOALLOC_SCRATCH_BYTES
 * (roughly nnz / 64 * (12 F + 12) bytes; about 340 thousand edges at
 * F = 128 fp32); larger problems are rejected with GNN_ERR_WORKSPACE before
 * any launch.  Other arguments, validation and errors are as for
 * gnn_segment_reduce_sum, and are checked first, in the same order and with
 * the same codes: a call rejected on the host touches neither the array nor
 * the stream.  n_rows == 0 returns GNN_OK with nothing launched.
 *
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) and caches it per device
 * ordinal; make that first call before any stream capture.  The cached
 * address does not survive cudaDeviceReset: do not call this entry point on
 * a device after resetting it in the same process.  X, Y and `stream` must
 * belong to the current device.  Each call clears the part of the
 * array it uses (cudaMemsetAsync on `stream`) before its kernel runs.  All
 * calls on a device share the one array, which keeps the last call's
 * contents: calls that may overlap on the GPU (different streams without
 * ordering between them) race on it and give wrong results. */
#define GNN_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
gnn_status gnn_segment_reduce_sum_noalloc(const gnn_csr *g, const void *prep, const void *X,
                                          int32_t x_dtype, int32_t F, float *Y, void *stream);

/* Y[i,:] = (sum over j in N(i) of X[j,:]) / d_in(i); empty rows give 0. */
gnn_status gnn_segment_reduce_mean(const gnn_csr *g, const void *prep, const void *X,
                                   int32_t x_dtype, int32_t F, float *Y, void *ws,
                                   size_t ws_bytes, void *stream);

/* Y[i,f] = max over j in N(i) of X[j,f] under the order-preserving key of
 * IO-aware GNN layers, Appendix D.1 (so -0 < +0); ties go to the smallest
 * source id.  argmax[i,f] (int32 [n_rows, F], may be NULL) = that source
 * node id (not an edge position).  Empty rows give Y = 0, argmax = -1.
 * Inputs must be finite.  Bit-exact. */
gnn_status gnn_segment_reduce_max(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, int32_t *argmax,
                                  void *ws, size_t ws_bytes, void *stream);

/* Y[i,f] = min over j in N(i) of X[j,f], argmin[i,f] = that j: the min
 * reduction with argmin of IO-aware GNN layers, Appendix D.1.  Values are
 * compared through the order-preserving key (so -0 < +0), ties go to the
 * smallest source id, and cut rows merge a packed (key, index) word, so the
 * result is exact and deterministic.  Empty rows give 0 and argmin -1.
 * argmin may be NULL.  Shapes and F as gnn_spmm; workspace
 * gnn_workspace_size(GNN_OP_MIN, ...). */
gnn_status gnn_segment_reduce_min(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, int32_t *argmin,
                                  void *ws, size_t ws_bytes, void *stream);

/* Backward of gnn_segment_reduce_max / _min (IO-aware GNN layers, Appendix
 * D.1: the gradient flows only along the stored argmin / argmax, a sparse
 * scatter-add): grad_X[arg[v,f], f] += grad_out[v,f] for every v, f with
 * arg[v,f] >= 0.  arg int32 and grad_out fp32 are [n_rows, F]; grad_X fp32
 * [n_cols, F] is overwritten (zero-filled first).  F % 4 == 0 (else
 * GNN_ERR_UNSUPPORTED), every pointer 16-byte aligned.  fp32 atomic adds:
 * sums of several gradients into one entry round in arrival order.  An arg
 * >= n_cols sets the device error word (GNN_ERR_DEVICE_CHECK) and is
 * skipped.  No workspace.  Asynchronous. */
gnn_status gnn_segment_reduce_ext_backward(const int32_t *arg, int32_t n_rows, int32_t F,
                                           const float *grad_out, int32_t n_cols, float *grad_X,
                                           void *stream);

/* -------------------------------------------- step a3: dense projection */

/* C = H W  (IO-aware GNN layers, Section 2.2 (i), the dense GEMM of
 * footnote 2).  H [n, F_in], W [F_in, F_out] row-major, C [n, F_out].
 * bf16 inputs: tcgen05 tensor cores, fp32 accumulation in TMEM, C bf16;
 * F_in % 64 == 0, F_out % 16 == 0, F_out <= 256.  fp32 inputs: fp32 FMA
 * (no TF32), C fp32. */
gnn_status gnn_projection(const void *H, int32_t dtype, int64_t n, int32_t F_in, const void *W,
                          int32_t F_out, void *C, void *stream);

/* ------------------------------------------------ step a4: fused GATv2 */

/* GATv2 forward (IO-aware GNN layers, Section 2.2 (iii); Appendix D.2 fused
 * CSR forward): l = H W_l, r = H W_r (W_r NULL: shared W, l = r), then per
 * destination i and head h
 *   e_ij = sum_d a[h,d] LeakyReLU_neg_slope(l[i,h,d] + r[j,h,d]),
 *   out[i,h,:] = sum_j softmax_j(e_ij) r[j,h,:],
 *   lse[i,h] = ln sum_j exp(e_ij)   (lse may be NULL).
 * Score, online softmax and aggregation run in one pass; no per-edge tensor
 * is written.  H [n_cols, F_in]; W [F_in, heads*head_dim]; a fp32 [heads,
 * head_dim]; out fp32 [n_rows, heads*head_dim]; lse fp32 [n_rows, heads].
 * dtype bf16: projections on tcgen05, l/r stored bf16 in ws.  dtype fp32:
 * fp32 projections.  head_dim in {32, 64, 128}; heads*head_dim <= 256
 * (bf16) or <= 1024 (fp32); square graphs only.  Empty rows give out 0,
 * lse -inf. */
gnn_status gnn_gatv2_fwd(const gnn_csr *g, const void *prep, const void *H, int32_t dtype,
                         int32_t F_in, const void *W_l, const void *W_r, const float *a,
                         int32_t heads, int32_t head_dim, float neg_slope, float *out,
                         float *lse, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------- step a6: block-sparse tiles */

/* Block-sparse tile layout (IO-aware GNN layers, Section 3.3 and Appendix
 * D.3, weighted block-sparse format): rows are cut into 16-row windows and
 * 128-row groups (8 windows).  U_g = sorted unique source columns of group
 * g; column block b = U_g[16b .. 16b+16) (padding entries are column 0 and
 * never masked in).  Tile (window w, block b) is 16x16 with a 256-bit mask,
 * bit r*16+c (word (r*16+c)/64) set iff edge U_g[16b+c] -> 16w+r exists.
 * A tile is kept iff popcount >= 1 and popcount/256 >= fill_threshold (fp32
 * comparison); a block is listed iff one of its 8 tiles is kept; masks of
 * unkept tiles are zero; edges of unkept tiles form the residual CSR. */
typedef struct {
    int32_t n_rows, n_groups;
    int64_t n_blocks;        /* listed column blocks */
    int64_t n_tiles_kept;    /* kept 16x16 tiles */
    int64_t nnz_tiles;       /* edges inside kept tiles */
    int64_t nnz_residual;    /* edges in the residual CSR */
    float fill_threshold;
    int32_t packing;         /* gnn_packing the plan was made with */
    /* device pointers into the caller's buffer */
    int32_t *grp_blk_offset; /* [n_groups+1] */
    int32_t *blk_cols;       /* [n_blocks*16] */
    uint64_t *blk_mask;      /* [n_blocks*8*4] */
    int32_t *res_rowptr;     /* [n_rows+1] */
    int32_t *res_colidx;     /* [nnz_residual] */
} gnn_blocksparse;

/* Order of a group's columns before they are cut into 16-column blocks.
 * GNN_PACK_ID: ascending source id (the pages' "sorted" columns).
 * GNN_PACK_COUNT: descending number of the group's edges from that source,
 * ties by ascending id, which gathers the busiest columns into the first
 * blocks and raises their tiles' fill (IO-aware GNN layers, Appendix D.3,
 * columns packed into tensor-core blocks).  Everything else in the layout is
 * as above, with U_g taken in the packed order. */
typedef enum { GNN_PACK_ID = 0, GNN_PACK_COUNT = 1 } gnn_packing;

/* Synchronous planning pass: fills the counts of *bs (host struct; pointers
 * left NULL) and *out_bytes, the size of the buffer gnn_blocksparse_build
 * needs.  fill_threshold in [0, 1].  Columns in id order (GNN_PACK_ID). */
gnn_status gnn_blocksparse_plan(const gnn_csr *g, float fill_threshold, void *ws,
                                size_t ws_bytes, gnn_blocksparse *bs, size_t *out_bytes,
                                void *stream);

/* As gnn_blocksparse_plan, with the column packing chosen (gnn_packing; any
 * other value is GNN_ERR_INVALID_ARG).  The plan records it in bs->packing,
 * which gnn_blocksparse_build follows.  Same workspace. */
gnn_status gnn_blocksparse_plan_packed(const gnn_csr *g, float fill_threshold, int32_t packing,
                                       void *ws, size_t ws_bytes, gnn_blocksparse *bs,
                                       size_t *out_bytes, void *stream);

/* Build the layout planned by gnn_blocksparse_plan into `out` (device,
 * out_bytes, 256-byte aligned); sets the device pointers of *bs (host struct).
 * If the graph's counts differ from the plan's, returns GNN_ERR_INVALID_ARG
 * and writes nothing to `out`.  Bit-exact.  Synchronous.  ws: as for the
 * plan, gnn_workspace_size(GNN_OP_BLOCKSPARSE, g, 0, 0, 0) bytes. */
gnn_status gnn_blocksparse_build(const gnn_csr *g, gnn_blocksparse *bs, void *out,
                                 size_t out_bytes, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------- steps a5 + a7: Graph Transformer attention */

/* GCN SpMM (as gnn_spmm, mapping aside) over a block-sparse layout from
 * gnn_blocksparse_build: the kept 16x16 tiles on the tensor cores
 * (tcgen05, bf16 operands, fp32 accumulation in TMEM), the residual edges on
 * the CSR SpMM, the two results added (IO-aware GNN layers, Section 3.3 and
 * Appendix D.3, the weighted block-sparse SpMM).  Each normalisation is a
 * row factor times a column factor from the whole graph's degrees; inside a
 * tile the column factor is rounded to bf16.  X bf16 [n_cols, F] with F a
 * multiple of 64; Y fp32 [n_rows, F]; graphs with edge values are not
 * supported (GNN_ERR_UNSUPPORTED).  prep required unless norm is NONE.
 * Workspace gnn_workspace_size(GNN_OP_SPMM_BLOCKSPARSE, g, F, 0, 0). */
gnn_status gnn_spmm_blocksparse(const gnn_csr *g, const void *prep, const gnn_blocksparse *bs,
                                int32_t norm, const void *X, int32_t x_dtype, int32_t F, float *Y,
                                void *ws, size_t ws_bytes, void *stream);

/* Graph Transformer attention (IO-aware GNN layers, Section 2.2 (iii);
 * Appendix D.2 fused CSR forward; Appendix D.3 tensor-core attention):
 *   e_ij = scale * sum_d Q[i,h,d] K[j,h,d]  (query at the destination),
 *   out[i,h,:] = sum_j softmax_j(e_ij) V[j,h,:], lse[i,h] = ln sum_j exp(e_ij).
 * bs NULL: fused CSR kernel over g.  bs from gnn_blocksparse_build on g:
 * edges in kept tiles run on tcgen05 (S = Q K^T and P V per 128-row group),
 * residual edges on the CSR kernel, softmax states merged.  Q, K, V
 * [n, heads*head_dim] (bf16 for the tile path; fp32 or bf16 for CSR), out
 * fp32 [n_rows, heads*head_dim], lse fp32 [n_rows, heads] (may be NULL).
 * head_dim in {32, 64}; square graphs. */
gnn_status gnn_gt_attn_fwd(const gnn_csr *g, const void *prep, const gnn_blocksparse *bs,
                           const void *Q, const void *K, const void *V, int32_t dtype,
                           int32_t heads, int32_t head_dim, float scale, float *out,
                           float *lse, void *ws, size_t ws_bytes, void *stream);

/* Backward of gnn_gt_attn_fwd on the CSR path (IO-aware GNN layers,
 * Appendix D.2: Delta = <O, dO> per destination and head, then the weights
 * recomputed from the stored logsumexp, dQ over the CSR and dK, dV over
 * CSR^T; no atomics on gradients, deterministic).  Graphs of mean degree 32
 * or more give each gradient row one warp; sparser (power-law) graphs run
 * warps over 256-edge runs, a row longer than a run cut into pieces that the
 * last to finish sums in edge order.
 * g square; gt its transpose from gnn_csr_transpose (rows = sources).
 * Q, K, V bf16 [n, heads*head_dim] as in the forward; out, lse (natural
 * log) from the forward; dout fp32 [n, heads*head_dim]; dQ, dK, dV fp32
 * [n, heads*head_dim], overwritten.  heads*head_dim in {128, 256} and
 * head_dim a power-of-two multiple of heads*head_dim/32 (else
 * GNN_ERR_UNSUPPORTED).  Workspace gnn_workspace_size(GNN_OP_GT_BACKWARD,
 * g, 0, heads, head_dim).  Asynchronous. */
gnn_status gnn_gt_attn_bwd(const gnn_csr *g, const gnn_csr *gt, const void *Q, const void *K,
                           const void *V, int32_t dtype, int32_t heads, int32_t head_dim, float scale,
                           const float *out, const float *lse, const float *dout, float *dQ, float *dK,
                           float *dV, void *ws, size_t ws_bytes, void *stream);

/* Backward of the GATv2 attention with respect to its per-node features and
 * its attention vector (IO-aware GNN layers, Appendix D.2, the GATv2
 * backward: an AL kernel over the CSR for the left features and the
 * attention vector, with G_i = sum_j alpha_ij <dO_i, r_j>, an R kernel over
 * CSR^T for the right features, and a reduction of the attention-vector
 * gradient over the nodes).  With x_ij = l_i + r_j per head, sigma =
 * LeakyReLU(neg_slope), e_ij = <a_h, sigma(x_ij)> and alpha_ij =
 * exp(e_ij - lse_i):
 *   de_ij = alpha_ij (<dO_i, r_j> - G_i)
 *   dl_i = sum_j de_ij a_h . sigma'(x_ij),  da_h = sum_ij de_ij sigma(x_ij),
 *   dr_j = sum_i alpha_ij dO_i + de_ij a_h . sigma'(x_ij).
 * G_i is computed as <out_i, dout_i> (equal, since out_i = sum_j alpha_ij
 * r_j).  Cl (l, destination side) and Cr (r, source side) are the projected
 * features [n, heads*head_dim] the forward scored, fp32 or bf16 (dtype);
 * with one projection (W_r = W_l) pass the same C for both, and its
 * gradient is dl + dr.  The gradient through the projection itself (dW =
 * H^T dC, dH = dC W^T) is a dense GEMM left to the caller.  a fp32
 * [heads, head_dim]; out, lse from gnn_gatv2_fwd; dout fp32; dl, dr fp32
 * [n, heads*head_dim] and da fp32 [heads*head_dim], overwritten.  g square,
 * gt its transpose (gnn_csr_transpose).  heads*head_dim in {32, 64, 128,
 * 256}; with c = heads*head_dim/32 channels per lane, head_dim must be a
 * power-of-two multiple of c (else GNN_ERR_UNSUPPORTED).  Rows are worked in runs of 256 edges with heavy
 * rows cut and their pieces summed in edge order: deterministic.  Workspace
 * gnn_workspace_size(GNN_OP_GATV2_BACKWARD, g, 0, heads, head_dim), any
 * contents (the call clears what it needs).  Asynchronous. */
gnn_status gnn_gatv2_attn_bwd(const gnn_csr *g, const gnn_csr *gt, const void *Cl, const void *Cr,
                              int32_t dtype, const float *a, int32_t heads, int32_t head_dim,
                              float neg_slope, const float *out, const float *lse,
                              const float *dout, float *dl, float *dr, float *da, void *ws,
                              size_t ws_bytes, void *stream);

/* ------------------------------------------- adaptive choice of backend */

/* Graph statistics an adaptive runtime chooses backends from (IO-aware GNN
 * layers, Section 5: degree skew, local density, feature size; Appendix
 * B.1, Table 5's degree skewness).  Degrees are row lengths (in-degrees);
 * moments are population moments: skewness = m3 / m2^(3/2), 0 when m2 = 0.
 * n_blocks: 128 x 16 column blocks holding at least one edge (the
 * block-sparse plan at fill 0); edges_per_block = nnz / n_blocks, the local
 * density the tensor-core tiles depend on. */
typedef struct {
    int32_t n_rows;
    int64_t nnz;
    int32_t max_degree;
    double mean_degree, degree_std, degree_skewness;
    int64_t n_blocks;
    double edges_per_block;
} gnn_graph_stats;

typedef enum { GNN_BACKEND_CSR = 0, GNN_BACKEND_TILES = 1 } gnn_backend;

/* Measures *out on the GPU (one pass over rowptr, then the block-sparse
 * plan).  Synchronous: returns with *out filled.  Deterministic.  Workspace
 * gnn_workspace_size(GNN_OP_GRAPH_STATS, g, 0, 0, 0). */
gnn_status gnn_graph_stats_compute(const gnn_csr *g, gnn_graph_stats *out, void *ws,
                                   size_t ws_bytes, void *stream);

/* Host rule, no GPU work: the backend for op (GNN_OP_SPMM or GNN_OP_GT;
 * every other op has only the CSR kernels) on a graph with statistics *s,
 * features of `dtype` and width F (SpMM) or heads x head_dim (GT).  Tiles
 * need bf16, F % 64 == 0 (SpMM) or head_dim in {32, 64} (GT), and pay off
 * above a local density measured on GB300: 158 edges per listed block for
 * SpMM, 129 for GT (the tile rate in blocks/s against the CSR rate in
 * edges/s; both scale with the feature width alike).  *fill_threshold (may
 * be NULL) receives the threshold to build the tiles with: 0 (every edge in
 * a tile), the fastest setting measured.  Returns a gnn_backend. */
int32_t gnn_select_backend(const gnn_graph_stats *s, int32_t op, int32_t dtype, int32_t F,
                           int32_t heads, int32_t head_dim, float *fill_threshold);

/* --------------------------------------------------- step a8: reordering */

typedef enum { GNN_PERM_IDENTITY = 0, GNN_PERM_RANDOM = 1, GNN_PERM_DEGREE = 2,
               GNN_PERM_RCM = 3 } gnn_perm_kind;

/* Vertex ordering of a square graph (IO-aware GNN layers, Section 2.4 and
 * Section 4.1; RCM per the marginalized-graph-kernel solver's reordering
 * section).  perm[new] = old, inv[old] = new (either may be NULL).
 *   RANDOM: ascending (splitmix64(seed ^ id), id)
 *   DEGREE: descending d_in + d_out (as stored), ties by ascending id
 *   RCM:    reverse Cuthill-McKee on A + A^T without self-loops; each
 *           component starts at its unvisited node of smallest degree
 *           (lowest id), each visited node appends its unvisited neighbours
 *           in ascending (degree, id).
 * Bit-exact.  IDENTITY/RANDOM/DEGREE are asynchronous; RCM is synchronous
 * (its number of breadth-first levels is data dependent). */
gnn_status gnn_reorder_perm(const gnn_csr *g, int32_t kind, uint64_t seed, int32_t *perm,
                            int32_t *inv, void *ws, size_t ws_bytes, void *stream);

/* Relabel: new row r = old row perm[r] with columns mapped through inv and
 * re-sorted; rowptr_out [n+1], colidx_out [nnz]; if X is not NULL, X_out[r]
 * = X[perm[r]] ([n, F], x_dtype).  Bit-exact.  Asynchronous. */
gnn_status gnn_apply_perm(const gnn_csr *g, const int32_t *perm, const int32_t *inv,
                          int32_t *rowptr_out, int32_t *colidx_out, const void *X,
                          int32_t x_dtype, int32_t F, void *X_out, void *ws, size_t ws_bytes,
                          void *stream);

/* CSR^T (the CSR-transpose build the backward passes need): the graph with
 * every edge j -> i turned into i -> j, as a CSR by (former) source
 * (IO-aware GNN layers, Appendix D.2, backward kernels over CSR^T).
 * rowptr_t [n_cols + 1], colidx_t [nnz]: row j of the result lists the i
 * with j in N(i), ascending; values_t [nnz] (may be NULL; requires
 * g->values) carries each edge's value.  The backward of gnn_spmm is a
 * gnn_spmm on the result: GCN (BOTH) as is (the transposed graph's prepared
 * degrees swap roles), plain sum with NONE, mean with RIGHT.  Workspace
 * gnn_workspace_size(GNN_OP_TRANSPOSE, g, 0, 0, 0).  Asynchronous. */
gnn_status gnn_csr_transpose(const gnn_csr *g, int32_t *rowptr_t, int32_t *colidx_t, float *values_t,
                             void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------ utilities */

const char *gnn_status_string(int32_t status);
/* Number of kernels this library has launched in this process (host
 * counter, incremented at every launch). */
uint64_t gnn_launch_count(void);
/* Library version string. */
const char *gnn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GNN_H */
