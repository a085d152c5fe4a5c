// Step a7: Graph Transformer attention over the kept 16x16 tiles of a
// block-sparse layout on the 5th-generation tensor cores, merged with the
// fused CSR attention over the residual edges.
//
// IO-aware GNN layers, Section 3.3 and Appendix D.3 (tensor-core attention on
// the weighted block-sparse format: per row window, scores against the packed
// column tiles, the tile bitmaps masking absent edges, softmax and the
// weighted sum of values; the edges left out of the tiles go through the CSR
// kernel and the two softmax states are merged).
//
// GB300 design.  One CTA (4 warps, one thread per row) per 128-row group and
// head.  The group's listed column blocks are taken in chunks of up to
// kChunkBlocks blocks:
//   1. the chunk's K rows and V rows (head h) are gathered into shared memory
//      in the no-swizzle core-matrix layout of tcgen05 operands (8 rows x 16
//      bytes per core matrix), every load of the chunk issued before the
//      first store; V is written transposed so that both operands of the
//      second product are K-major; each thread fetches its row's tile-mask
//      bits for the chunk alongside;
//   2. one thread issues S = Q K^T (M = 128, N = 16 x blocks, K = head_dim)
//      into TMEM;
//   3. each thread reads its row of S (tcgen05.ld), masks it with the tile
//      bitmaps, updates its online-softmax state (running max, running sum,
//      rescale of its output row) and writes P = exp(S - m) in bf16 to
//      shared memory;
//   4. one thread issues O_chunk = P V (M = 128, N = head_dim, K = columns);
//      each thread adds its row of O_chunk to its output row in registers.
// The residual edges run first on the CSR kernel, which writes (out, lse);
// the tile state is then merged with it through the logsumexp.  With no
// residual edges the tile kernel writes every row itself (empty rows: 0 and
// lse = -inf), so out is neither pre-written nor read back.  MMA
// completion is tracked with an mbarrier; every wait is bounded.
#include <algorithm>
#include <mutex>

#include "async.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

extern "C" gnn_status gnn_gt_attn_fwd(const gnn_csr *g, const void *prep, const gnn_blocksparse *bs,
                                      const void *Q, const void *K, const void *V, int32_t dtype,
                                      int32_t heads, int32_t head_dim, float scale, float *out, float *lse,
                                      void *ws, size_t ws_bytes, void *stream);

namespace gnn {

size_t gt_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim);

namespace {

constexpr int kRows = 128;          // rows per group (MMA M)
// Column blocks per chunk: S takes 16 per block TMEM columns and O the next
// D, within a power-of-two allocation.  128 columns per CTA let four CTAs
// share an SM's 512; measured on GB300 (GT at c4, D = 32, tiles at fill >=
// 0.2): 12 blocks 1.23 ms, 8 1.12, 6 0.85, 4 0.88.
__host__ __device__ constexpr int chunk_blocks(int D) { return D == 32 ? 6 : 4; }
__host__ __device__ constexpr int o_col(int D) { return chunk_blocks(D) * 16; }
__host__ __device__ constexpr int tmem_cols_for(int n) { return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256; }
constexpr float kLog2eT = 1.4426950408889634f;
constexpr float kLn2T = 0.6931471805599453f;
// lazy-rescale margin of the tile softmax (base-2 units), as in the CSR kernels
constexpr float kLazyT = 8.f;

struct TileArgs {
    const int32_t *grp_blk_offset;
    const int32_t *blk_cols;
    const unsigned long long *blk_mask;
    const __nv_bfloat16 *Q, *K, *V;
    float *out;        // holds the residual result on entry
    float *lse;        // [n, heads]: the residual logsumexp on entry, the merged one on exit
    int32_t n_rows, heads, D;
    int32_t has_residual;  // 0: no residual edges; out and lse are written here, not merged
    float qscale;      // scale * log2 e
    int32_t *err;
};

__device__ __forceinline__ void st16s(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

template <int D>
__global__ void __launch_bounds__(kRows) k_gt_tiles(TileArgs t) {
    constexpr int kChunkBlocks = chunk_blocks(D);
    constexpr int kOCol = o_col(D);
    constexpr int kTmemCols = tmem_cols_for(kOCol + D);
    static_assert(kOCol + D <= 256, "S and O must fit one 256-column allocation");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~(uintptr_t)1023);
    constexpr int NCMAX = kChunkBlocks * 16;
    unsigned char *sQ = base;                         // [16][D/8] core matrices
    unsigned char *sK = sQ + kRows * D * 2;           // [NC/8][D/8]
    unsigned char *sV = sK + NCMAX * D * 2;           // [D/8][NC/8] (V transposed), padded rows
    unsigned char *sP = sV + NCMAX * D * 2 + (D / 8) * 16;  // [16][NC/8]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sP + kRows * NCMAX * 2);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);

    // heads vary fastest: the CTAs of one group run close together, so each
    // gathered K / V row is fetched from DRAM once and its other heads'
    // slices are still in L2 when their CTAs read them (0.621 -> 0.586 ms on
    // the clustered graph at fill 0)
    const int h = (int)(blockIdx.x % (unsigned)t.heads), g = (int)(blockIdx.x / (unsigned)t.heads);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int b0 = __ldg(t.grp_blk_offset + g), b1 = __ldg(t.grp_blk_offset + g + 1);
    const int64_t HD = (int64_t)t.heads * D;
    const int32_t row = g * kRows + tid;
    const bool valid = row < t.n_rows;
    if (b0 == b1) {
        // no tiles: the residual result stands, or (no residual) the rows are empty
        if (!t.has_residual && valid) {
            float *orow = t.out + (int64_t)row * HD + h * D;
#pragma unroll
            for (int d = 0; d < D; d += 4) *reinterpret_cast<float4 *>(orow + d) = make_float4(0.f, 0.f, 0.f, 0.f);
            t.lse[(int64_t)row * t.heads + h] = -INFINITY;
        }
        return;
    }

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    // Q tile: row tid, dims [8k, 8k+8) -> core matrix (tid/8, k)
#pragma unroll
    for (int k = 0; k < D / 8; ++k) {
        const uint4 v = valid ? ldg16(t.Q + row * HD + h * D + 8 * k) : make_uint4(0u, 0u, 0u, 0u);
        st16s(sQ + ((tid / 8) * (D / 8) + k) * 128 + (tid % 8) * 16, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t idesc_o = bf16_idesc(kRows, D);

    float m = -INFINITY, l = 0.f;
    float o[D];
#pragma unroll
    for (int d = 0; d < D; ++d) o[d] = 0.f;
    uint32_t phase = 0;
    bool ok = true;
    const int w = (tid % kRows) / 16, r = tid % 16;  // window and row within it

    for (int c0 = b0; c0 < b1 && ok; c0 += kChunkBlocks) {
        const int nbk = min(kChunkBlocks, b1 - c0);
        const int NC = nbk * 16;
        // this row's mask bits of the chunk's blocks (16 per block), fetched
        // together ahead of the gather
        uint32_t mk[(kChunkBlocks + 1) / 2];
        {
            unsigned long long mw[kChunkBlocks];
#pragma unroll
            for (int b = 0; b < kChunkBlocks; ++b)
                mw[b] = b < nbk ? __ldg(t.blk_mask + ((int64_t)(c0 + b) * 8 + w) * 4 + (r * 16) / 64) : 0ull;
#pragma unroll
            for (int b = 0; b < kChunkBlocks; b += 2) {
                const uint32_t lo = (uint32_t)(mw[b] >> ((r * 16) % 64)) & 0xFFFFu;
                const uint32_t hi = b + 1 < kChunkBlocks ? (uint32_t)(mw[b + 1] >> ((r * 16) % 64)) & 0xFFFFu : 0u;
                mk[b / 2] = lo | (hi << 16);
            }
        }
        // V^T rows of core matrices are (NC/8)*128 + 16 bytes apart: the
        // 16-byte pad puts the four channel groups that a warp writes at once
        // in different shared-memory banks
        const int vstride = (NC / 8) * 128 + 16;
        // gather K (as rows) and V (transposed) of the chunk's columns: all
        // column ids first, then all rows, then the shared-memory stores
        constexpr int IT = NCMAX * (D / 8) / kRows;
        static_assert(NCMAX * (D / 8) % kRows == 0, "the gather covers a chunk in whole rounds");
        int32_t colv[IT];
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kRows;
            colv[i] = idx < NC * (D / 8) ? __ldg(t.blk_cols + (int64_t)c0 * 16 + idx / (D / 8)) : 0;
        }
        uint4 kvv[IT], vvv[IT];
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kRows;
            if (idx < NC * (D / 8)) {
                const int k = idx % (D / 8);
                kvv[i] = ldg16(t.K + (int64_t)colv[i] * HD + h * D + 8 * k);
                vvv[i] = ldg16(t.V + (int64_t)colv[i] * HD + h * D + 8 * k);
            }
        }
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kRows;
            if (idx < NC * (D / 8)) {
                const int c = idx / (D / 8), k = idx % (D / 8);
                st16s(sK + ((c / 8) * (D / 8) + k) * 128 + (c % 8) * 16, kvv[i]);
                const uint16_t *ve = reinterpret_cast<const uint16_t *>(&vvv[i]);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int d = 8 * k + q;
                    *reinterpret_cast<uint16_t *>(sV + (d / 8) * vstride + (c / 8) * 128 + (d % 8) * 16 +
                                                  (c % 8) * 2) = ve[q];
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // S = Q K^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_bf16(tmem, plain_desc(su32(sQ) + ks * 256, 128, (D / 8) * 128),
                          plain_desc(su32(sK) + ks * 256, 128, (D / 8) * 128), bf16_idesc(kRows, NC), ks > 0);
            umma_commit(bar);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar, phase))) {
            ok = false;
            break;
        }
        phase ^= 1u;
        tc_fence_after();
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        // P = exp2(s - m) (0 where masked) into shared memory, its rounded
        // weights summed into l; with track, also the chunk's masked maximum
        // (scores in base-2 units) in cm
        auto exp_pass = [&](bool write, bool track, float &cm) {
#pragma unroll
            for (int cc = 0; cc < NCMAX; cc += 32) {
                if (cc >= NC) break;
                uint32_t v[32];
                tmem_ld32(lane_base + (uint32_t)cc, v);
                const uint32_t mkc = (cc + 16 < NC) ? mk[cc / 32] : (mk[cc / 32] & 0xFFFFu);
                const int nq = min(32, NC - cc);
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    if (g8 * 8 >= nq) break;
                    uint32_t pk[4];
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        const int q = g8 * 8 + 2 * q2;
                        const bool b0 = (mkc >> q) & 1u, b1 = (mkc >> (q + 1)) & 1u;
                        const float s0 = __uint_as_float(v[q]) * t.qscale;
                        const float s1 = __uint_as_float(v[q + 1]) * t.qscale;
                        if (track) {
                            if (b0) cm = fmaxf(cm, s0);
                            if (b1) cm = fmaxf(cm, s1);
                        }
                        const float p0 = b0 ? exp2_approx(s0 - m) : 0.f;
                        const float p1 = b1 ? exp2_approx(s1 - m) : 0.f;
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                        // the sum uses the rounded weights, the ones the product uses
                        if (write) l += __low2float(b2) + __high2float(b2);
                        pk[q2] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    const int c = cc + g8 * 8;
                    if (write)
                        st16s(sP + ((tid / 8) * (NC / 8) + c / 8) * 128 + (tid % 8) * 16,
                              make_uint4(pk[0], pk[1], pk[2], pk[3]));
                }
            }
        };
        // One pass when every row of the warp has a running maximum: P is
        // formed against it while the chunk maximum is taken alongside, and a
        // row keeps that P unless its chunk maximum passes the running one by
        // more than kLazyT (weights then stay below 2^kLazyT).  Such rows, and
        // every row in its first chunk, take two passes: the masked maximum,
        // the rescale of l and o, then P.
        bool redo = true;
        if (__all_sync(0xffffffffu, m != -INFINITY)) {
            float cm = -INFINITY;
            const float l0 = l;
            exp_pass(true, true, cm);
            redo = cm > m + kLazyT;
            if (redo) l = l0;
        }
        if (__any_sync(0xffffffffu, redo)) {
            float cm = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < NCMAX; cc += 32) {
                if (cc >= NC) break;
                uint32_t v[32];
                tmem_ld32(lane_base + (uint32_t)cc, v);
                const uint32_t mkc = (cc + 16 < NC) ? mk[cc / 32] : (mk[cc / 32] & 0xFFFFu);
#pragma unroll
                for (int q = 0; q < 32; ++q)
                    if ((mkc >> q) & 1u) cm = fmaxf(cm, __uint_as_float(v[q]) * t.qscale);
            }
            if (redo) {
                const float mn = fmaxf(m, cm);
                const float sc = (m == -INFINITY) ? 0.f : exp2_approx(m - mn);
                l *= sc;
#pragma unroll
                for (int d = 0; d < D; ++d) o[d] *= sc;
                m = mn;
            }
            float unused = -INFINITY;
            exp_pass(redo, false, unused);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // O_chunk = P V
        if (tid == 0) {
            for (int ks = 0; ks < NC / 16; ++ks)
                umma_bf16(tmem + kOCol, plain_desc(su32(sP) + ks * 256, 128, (NC / 8) * 128),
                          plain_desc(su32(sV) + ks * 256, 128, vstride), idesc_o, ks > 0);
            umma_commit(bar);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar, phase))) {
            ok = false;
            break;
        }
        phase ^= 1u;
        tc_fence_after();
#pragma unroll
        for (int d0 = 0; d0 < D; d0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_base + (uint32_t)(kOCol + d0), v);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[d0 + q] += __uint_as_float(v[q]);
        }
        tc_fence_before();
        __syncthreads();  // the next chunk overwrites sK, sV, sP and S
        tc_fence_after();
    }
    if (!ok) {
        set_device_error(t.err, GNN_ERR_TIMEOUT);
        // an MMA still in flight completes before TMEM is released
        mbar_wait_bounded(bar, phase);
    }
    if (ok && valid && !t.has_residual) {
        // no residual edges: this is the whole result
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float *orow = t.out + (int64_t)row * HD + h * D;
#pragma unroll
        for (int d = 0; d < D; d += 4)
            *reinterpret_cast<float4 *>(orow + d) = make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
        t.lse[(int64_t)row * t.heads + h] = l > 0.f ? (m + log2f(l)) * kLn2T : -INFINITY;
    }
    // merge with the residual CSR result (out, lse_res) through the logsumexp
    if (ok && valid && t.has_residual && l > 0.f) {
        const float lse_t = (m + log2f(l)) * kLn2T;
        const float lse_r = t.lse[(int64_t)row * t.heads + h];
        const float L = lse_r == -INFINITY ? lse_t : fmaxf(lse_r, lse_t) + log1pf(expf(-fabsf(lse_r - lse_t)));
        const float cr = lse_r == -INFINITY ? 0.f : expf(lse_r - L);
        const float ct = expf(lse_t - L) / l;
        float *orow = t.out + (int64_t)row * HD + h * D;
#pragma unroll
        for (int d = 0; d < D; d += 4) {
            const float4 rv = *reinterpret_cast<const float4 *>(orow + d);
            *reinterpret_cast<float4 *>(orow + d) = make_float4(rv.x * cr + o[d] * ct, rv.y * cr + o[d + 1] * ct,
                                                                rv.z * cr + o[d + 2] * ct, rv.w * cr + o[d + 3] * ct);
        }
        t.lse[(int64_t)row * t.heads + h] = L;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// Dynamic shared memory per CTA: the operands, raised if needed so that no
// more CTAs are resident on an SM than its 512 TMEM columns serve (an extra
// one would only wait in tcgen05.alloc).
template <int D>
size_t tile_smem_bytes() {
    constexpr int kChunkBlocks = chunk_blocks(D);
    constexpr int kOCol = o_col(D);
    const size_t need = 1024 + (size_t)kRows * D * 2 + 2 * (size_t)kChunkBlocks * 16 * D * 2 + (D / 8) * 16 +
                        (size_t)kRows * kChunkBlocks * 16 * 2 + 64;
    const size_t ctas = 512 / tmem_cols_for(kOCol + D);
    const size_t floor = (size_t)228 * 1024 / (ctas + 1) - 1024 + 64;
    return std::max(need, floor);
}

template <int D>
cudaError_t launch_tiles(const TileArgs &t, int32_t n_groups, cudaStream_t s) {
    const cudaError_t attr = func_attr(reinterpret_cast<const void *>(k_gt_tiles<D>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (attr != cudaSuccess) return attr;
    k_gt_tiles<D><<<(unsigned)((int64_t)n_groups * t.heads), kRows, tile_smem_bytes<D>(), s>>>(t);
    return cudaGetLastError();
}

}  // namespace

// Workspace of the tile path: residual logsumexp, then the CSR workspace.
size_t gt_tiles_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim) {
    return round_up(sizeof(float) * (size_t)g->n_rows * heads, 256) + gt_workspace_bytes(g, heads, head_dim);
}

gnn_status gt_attn_tiles(const gnn_csr *g, const gnn_blocksparse *bs, const void *Q, const void *K, const void *V,
                         int32_t heads, int32_t head_dim, float scale, float *out, float *lse, void *ws,
                         size_t ws_bytes, cudaStream_t s) {
    if (head_dim != 32 && head_dim != 64) return GNN_ERR_UNSUPPORTED;
    if (!bs->grp_blk_offset || !bs->res_rowptr || bs->n_rows != g->n_rows) return GNN_ERR_INVALID_ARG;
    if (bs->n_groups != (g->n_rows + kRows - 1) / kRows) return GNN_ERR_INVALID_ARG;
    const size_t need = gt_tiles_workspace_bytes(g, heads, head_dim);
    if (!ws || ws_bytes < need) return GNN_ERR_WORKSPACE;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    // the residual logsumexp goes to the caller's lse (or the workspace) and
    // is merged there in place; rows without tiles keep it
    Carver cv(ws);
    float *lse_ws = cv.take<float>((size_t)g->n_rows * heads);
    float *lse_res = lse ? lse : lse_ws;
    void *csr_ws = static_cast<char *>(ws) + cv.used;
    // residual edges: fused CSR kernel, writing (out, lse_res); with no
    // residual edges (and some tiles) the tile kernel writes every row itself
    const bool has_residual = bs->nnz_residual > 0 || bs->n_blocks == 0;
    if (has_residual) {
        gnn_csr res{g->n_rows, g->n_cols, bs->nnz_residual, bs->res_rowptr, bs->res_colidx, nullptr};
        gnn_status st = gnn_gt_attn_fwd(&res, nullptr, nullptr, Q, K, V, GNN_BF16, heads, head_dim, scale, out,
                                        lse_res, csr_ws, ws_bytes - cv.used, s);
        if (st != GNN_OK) return st;
    }
    if (bs->n_blocks == 0) return GNN_OK;
    TileArgs t{};
    t.grp_blk_offset = bs->grp_blk_offset;
    t.blk_cols = bs->blk_cols;
    t.blk_mask = reinterpret_cast<const unsigned long long *>(bs->blk_mask);
    t.Q = static_cast<const __nv_bfloat16 *>(Q);
    t.K = static_cast<const __nv_bfloat16 *>(K);
    t.V = static_cast<const __nv_bfloat16 *>(V);
    t.out = out;
    t.lse = lse_res;
    t.n_rows = g->n_rows;
    t.heads = heads;
    t.D = head_dim;
    t.qscale = scale * kLog2eT;
    t.has_residual = has_residual ? 1 : 0;
    t.err = err;
    cudaError_t e = head_dim == 32 ? launch_tiles<32>(t, bs->n_groups, s) : launch_tiles<64>(t, bs->n_groups, s);
    note_launch();
    if (e != cudaSuccess) return cuda_status(e);
    return GNN_OK;
}

}  // namespace gnn
