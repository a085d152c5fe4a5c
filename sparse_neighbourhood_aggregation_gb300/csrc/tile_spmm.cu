// SpMM on the kept 16x16 tiles of a block-sparse layout with the
// 5th-generation tensor cores, the residual edges through the CSR SpMM.
//
// IO-aware GNN layers, Section 3.3 and Appendix D.3 (weighted block-sparse
// SpMM on tensor cores: per row window, the packed column tiles multiply the
// gathered feature rows, fp32 accumulation; the edges left out of the tiles
// go through the CSR kernel and the two results add).
//
// GB300 design.  Every normalisation of the GCN SpMM factors into a row
// factor times a column factor (NONE 1 x 1, LEFT 1/d_in(i) x 1, RIGHT
// 1 x 1/d_out(j), BOTH 1/sqrt(d_in(i)) x 1/sqrt(d_out(j)), degrees of the
// whole graph).  One CTA of 128 threads (one per row) takes a 128-row group
// and 64 features.  Per chunk of 6 column blocks (96 columns):
//   1. the chunk's feature rows are gathered, every load issued before the
//      first store, and written transposed into shared memory in the
//      no-swizzle core-matrix layout of a K-major tcgen05 operand; the
//      columns' factors go to shared memory alongside;
//   2. each thread writes its row of P = mask x column factor (bf16);
//   3. one thread issues O += P X (M = 128, N = 64, K = 96) into TMEM.
// O accumulates across chunks in TMEM with no rescaling; the epilogue reads
// it once, multiplies by the row factor and adds it to the residual result.
// Residual edges carry the full product of the two factors as edge values
// through the CSR SpMM.  MMA completion is tracked with an mbarrier; every
// wait is bounded.
#include <algorithm>

#include "async.cuh"
#include "common.cuh"
#include "tcgen05.cuh"

namespace gnn {

void prep_pointers(const gnn_csr *g, const void *prep, const int32_t **d_out, const float **dinv_in,
                   const float **dinv_out);
gnn_status check_csr_args(const gnn_csr *g);
size_t agg_workspace_bytes(const gnn_csr *g, int32_t op, int32_t x_dtype, int32_t F);

namespace {

constexpr int kTRows = 128;   // rows per group (MMA M)
constexpr int kTFeat = 64;    // features per CTA (MMA N, TMEM columns)
constexpr int kTBlocks = 6;   // column blocks per chunk
constexpr int kTCols = kTBlocks * 16;

struct TileSpmmArgs {
    const int32_t *grp_blk_offset;
    const int32_t *blk_cols;
    const unsigned long long *blk_mask;
    const __nv_bfloat16 *X;
    float *Y;             // holds the residual result on entry when has_residual
    const int32_t *rowptr, *d_out;
    const float *dinv_in, *dinv_out;
    int32_t n_rows, F, norm, has_residual;
    int32_t *err;
};

__device__ __forceinline__ float col_factor(const TileSpmmArgs &t, int32_t j) {
    if (t.norm == GNN_NORM_RIGHT) {
        const int32_t d = __ldg(t.d_out + j);
        return d > 0 ? __frcp_rn((float)d) : 0.f;
    }
    if (t.norm == GNN_NORM_BOTH) return __ldg(t.dinv_out + j);
    return 1.f;
}

__device__ __forceinline__ float row_factor_of(const TileSpmmArgs &t, int32_t i) {
    if (t.norm == GNN_NORM_LEFT) {
        const int32_t d = __ldg(t.rowptr + i + 1) - __ldg(t.rowptr + i);
        return d > 0 ? __frcp_rn((float)d) : 0.f;
    }
    if (t.norm == GNN_NORM_BOTH) return __ldg(t.dinv_in + i);
    return 1.f;
}

__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }

__global__ void __launch_bounds__(kTRows) k_spmm_tiles(TileSpmmArgs t) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                            ~(uintptr_t)1023);
    unsigned char *sP = base;                                        // [16][NC/8] core matrices
    unsigned char *sX = sP + kTRows * kTCols * 2;                    // [64/8][NC/8], padded rows
    float *sCF = reinterpret_cast<float *>(sX + (kTFeat / 8) * (kTCols / 8 * 128 + 16));
    uint64_t *bar = reinterpret_cast<uint64_t *>(sCF + kTCols);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);

    // feature blocks vary fastest: the CTAs of one group run close together,
    // so each gathered feature row is fetched from DRAM once
    const int nfb = t.F / kTFeat;
    const int g = (int)(blockIdx.x / (unsigned)nfb), f0 = (int)(blockIdx.x % (unsigned)nfb) * kTFeat;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t row = g * kTRows + tid;
    const bool valid = row < t.n_rows;
    const int b0 = __ldg(t.grp_blk_offset + g), b1 = __ldg(t.grp_blk_offset + g + 1);
    if (b0 == b1) {
        // no tiles: the residual result stands, or (no residual) the rows are 0
        if (!t.has_residual && valid) {
            float *y = t.Y + (int64_t)row * t.F + f0;
#pragma unroll
            for (int d = 0; d < kTFeat; d += 4) *reinterpret_cast<float4 *>(y + d) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(kTFeat));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t idesc = bf16_idesc(kTRows, kTFeat);
    const int w = tid / 16, r = tid % 16;  // window and row within it
    uint32_t phase = 0;
    bool ok = true;

    for (int c0 = b0; c0 < b1 && ok; c0 += kTBlocks) {
        const int nbk = min(kTBlocks, b1 - c0);
        const int NC = nbk * 16;
        // this row's mask bits of the chunk's blocks, fetched ahead of the gather
        uint32_t mk[kTBlocks / 2];
        {
            unsigned long long mw[kTBlocks];
#pragma unroll
            for (int b = 0; b < kTBlocks; ++b)
                mw[b] = b < nbk ? __ldg(t.blk_mask + ((int64_t)(c0 + b) * 8 + w) * 4 + (r * 16) / 64) : 0ull;
#pragma unroll
            for (int b = 0; b < kTBlocks; b += 2)
                mk[b / 2] = ((uint32_t)(mw[b] >> ((r * 16) % 64)) & 0xFFFFu) |
                            (((uint32_t)(mw[b + 1] >> ((r * 16) % 64)) & 0xFFFFu) << 16);
        }
        // gather the chunk's feature rows (features [f0, f0+64)) transposed:
        // X^T rows of core matrices are (NC/8)*128 + 16 bytes apart, the pad
        // spreading a warp's 2-byte stores over the banks
        const int xstride = (NC / 8) * 128 + 16;
        constexpr int IT = kTCols * (kTFeat / 8) / kTRows;
        static_assert(kTCols * (kTFeat / 8) % kTRows == 0, "the gather covers a chunk in whole rounds");
        int32_t colv[IT];
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kTRows;
            colv[i] = idx < NC * (kTFeat / 8) ? __ldg(t.blk_cols + (int64_t)c0 * 16 + idx / (kTFeat / 8)) : 0;
        }
        uint4 xv[IT];
        float cfv[IT];
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kTRows;
            if (idx < NC * (kTFeat / 8)) {
                const int k = idx % (kTFeat / 8);
                xv[i] = ldg16(t.X + (int64_t)colv[i] * t.F + f0 + 8 * k);
                cfv[i] = k == 0 ? col_factor(t, colv[i]) : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < IT; ++i) {
            const int idx = tid + i * kTRows;
            if (idx < NC * (kTFeat / 8)) {
                const int c = idx / (kTFeat / 8), k = idx % (kTFeat / 8);
                if (k == 0) sCF[c] = cfv[i];
                const uint16_t *xe = reinterpret_cast<const uint16_t *>(&xv[i]);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int n = 8 * k + q;
                    *reinterpret_cast<uint16_t *>(sX + (n / 8) * xstride + (c / 8) * 128 + (n % 8) * 16 + (c % 8) * 2) =
                        xe[q];
                }
            }
        }
        __syncthreads();  // sCF
        // this row of P: mask bit x column factor, bf16
        for (int c = 0; c < NC; c += 8) {
            uint32_t pk[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const int q = c + 2 * q2;
                const uint32_t m0 = (mk[q / 32] >> (q % 32)) & 1u, m1 = (mk[(q + 1) / 32] >> ((q + 1) % 32)) & 1u;
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(m0 ? sCF[q] : 0.f, m1 ? sCF[q + 1] : 0.f);
                pk[q2] = *reinterpret_cast<const uint32_t *>(&b2);
            }
            st16(sP + ((tid / 8) * (NC / 8) + c / 8) * 128 + (tid % 8) * 16, make_uint4(pk[0], pk[1], pk[2], pk[3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // O += P X
        if (tid == 0) {
            for (int ks = 0; ks < NC / 16; ++ks)
                umma_bf16(tmem, plain_desc(su32(sP) + ks * 256, 128, (NC / 8) * 128),
                          plain_desc(su32(sX) + ks * 256, 128, xstride), idesc, (c0 > b0 || ks > 0) ? 1u : 0u);
            umma_commit(bar);
        }
        // the next chunk overwrites sP, sX and sCF: wait for the MMAs
        if (!__syncthreads_and(mbar_wait_bounded(bar, phase))) {
            ok = false;
            break;
        }
        phase ^= 1u;
        tc_fence_after();
    }
    if (!ok) {
        set_device_error(t.err, GNN_ERR_TIMEOUT);
        mbar_wait_bounded(bar, phase);  // an MMA still in flight lands before TMEM is released
    } else {
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float o[kTFeat];
#pragma unroll
        for (int d0 = 0; d0 < kTFeat; d0 += 32) {
            uint32_t v[32];
            tmem_ld32(lane_base + (uint32_t)d0, v);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[d0 + q] = __uint_as_float(v[q]);
        }
        if (valid) {
            const float rf = row_factor_of(t, row);
            float *y = t.Y + (int64_t)row * t.F + f0;
#pragma unroll
            for (int d = 0; d < kTFeat; d += 4) {
                float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t.has_residual) res = *reinterpret_cast<const float4 *>(y + d);
                *reinterpret_cast<float4 *>(y + d) = make_float4(res.x + rf * o[d], res.y + rf * o[d + 1],
                                                                 res.z + rf * o[d + 2], res.w + rf * o[d + 3]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTFeat));
    }
}

constexpr size_t kTileSpmmSmem = 1024 + (size_t)kTRows * kTCols * 2 + (kTFeat / 8) * (kTCols / 8 * 128 + 16) +
                                 kTCols * 4 + 64;

// Residual edge values: the product of the whole graph's row and column
// factors (thread per residual row).
__global__ void k_residual_values(const int32_t *__restrict__ res_rowptr, const int32_t *__restrict__ res_colidx,
                                  TileSpmmArgs t, float *__restrict__ vals) {
    const int32_t stride = gridDim.x * blockDim.x;
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < t.n_rows; i += stride) {
        const int32_t b = res_rowptr[i], e = res_rowptr[i + 1];
        if (b == e) continue;
        const float rf = row_factor_of(t, i);
        for (int32_t k = b; k < e; ++k) vals[k] = rf * col_factor(t, res_colidx[k]);
    }
}

}  // namespace

size_t tile_spmm_workspace_bytes(const gnn_csr *g, int32_t F) {
    // residual values, then the CSR SpMM workspace sized for every edge
    return round_up(sizeof(float) * (size_t)std::max<int64_t>(g->nnz, 1), 256) +
           agg_workspace_bytes(g, GNN_OP_SPMM, GNN_BF16, F);
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_spmm_blocksparse(const gnn_csr *g, const void *prep, const gnn_blocksparse *bs,
                                           int32_t norm, const void *X, int32_t x_dtype, int32_t F, float *Y,
                                           void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!bs || !Y || (!X && g->n_cols > 0)) return GNN_ERR_INVALID_ARG;
    if (x_dtype != GNN_BF16 || F < kTFeat || F % kTFeat || g->values) return GNN_ERR_UNSUPPORTED;
    if (norm < GNN_NORM_NONE || norm > GNN_NORM_BOTH) return GNN_ERR_INVALID_ARG;
    if (norm != GNN_NORM_NONE && !prep) return GNN_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y)) return GNN_ERR_INVALID_ARG;
    if (!bs->grp_blk_offset || !bs->res_rowptr || bs->n_rows != g->n_rows ||
        bs->n_groups != (g->n_rows + kTRows - 1) / kTRows)
        return GNN_ERR_INVALID_ARG;
    const size_t need = tile_spmm_workspace_bytes(g, F);
    if (!ws || ws_bytes < need) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    if (g->n_rows == 0) return GNN_OK;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    cudaStream_t s = as_stream(stream);

    TileSpmmArgs t{};
    t.grp_blk_offset = bs->grp_blk_offset;
    t.blk_cols = bs->blk_cols;
    t.blk_mask = reinterpret_cast<const unsigned long long *>(bs->blk_mask);
    t.X = static_cast<const __nv_bfloat16 *>(X);
    t.Y = Y;
    t.rowptr = g->rowptr;
    if (prep) prep_pointers(g, prep, &t.d_out, &t.dinv_in, &t.dinv_out);
    t.n_rows = g->n_rows;
    t.F = F;
    t.norm = norm;
    t.err = err;
    // with no residual edges (and some tiles) the tile kernel writes every row
    t.has_residual = (bs->nnz_residual > 0 || bs->n_blocks == 0) ? 1 : 0;

    if (t.has_residual) {
        Carver cv(ws);
        float *vals = cv.take<float>((size_t)std::max<int64_t>(bs->nnz_residual, 1));
        void *agg_ws = static_cast<char *>(ws) + round_up(sizeof(float) * (size_t)std::max<int64_t>(g->nnz, 1), 256);
        const size_t agg_bytes = ws_bytes - round_up(sizeof(float) * (size_t)std::max<int64_t>(g->nnz, 1), 256);
        if (bs->nnz_residual > 0) {
            const int blocks = (int)std::min<int64_t>((g->n_rows + 255) / 256, (int64_t)sm_count() * 8);
            k_residual_values<<<blocks, 256, 0, s>>>(bs->res_rowptr, bs->res_colidx, t, vals);
            note_launch();
            GNN_LAUNCH_CHECK();
        }
        gnn_csr res{g->n_rows, g->n_cols, bs->nnz_residual, bs->res_rowptr, bs->res_colidx, vals};
        st = gnn_spmm(&res, nullptr, GNN_NORM_NONE, X, GNN_BF16, F, Y, GNN_MAP_AUTO, agg_ws, agg_bytes, stream);
        if (st != GNN_OK) return st;
    }
    if (bs->n_blocks == 0) return GNN_OK;
    k_spmm_tiles<<<(unsigned)((int64_t)bs->n_groups * (F / kTFeat)), kTRows, kTileSpmmSmem, s>>>(t);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}
