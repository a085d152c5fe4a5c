// Step a6: block-sparse tile layout of a CSR graph for tensor-core attention.
//
// IO-aware GNN layers, Section 3.3 and Appendix D.3 (weighted block-sparse
// format: row windows, the sorted unique source columns of a window packed
// into dense column tiles, a bitmap per tile, a fill-based choice between
// tensor-core tiles and the CSR path).  Layout (see gnn.h): 128-row groups
// of eight 16-row windows; U_g = sorted unique sources of group g; column
// block b = U_g[16b .. 16b+16) (padding = column 0, never masked in); tile
// (window w, block b) has mask bit r*16+c iff edge U_g[16b+c] -> 16w+r; a
// tile is kept iff popcount >= 1 and popcount/256 >= threshold (fp32); a
// block is listed iff one of its tiles is kept; edges of tiles not kept form
// the residual CSR.
//
// GB300 design.  One pass of device kernels and CUB sorts / scans:
//  1. keys (group << 32 | source) of all edges, radix-sorted; first
//     occurrences give U_g (unique flags + exclusive scan) and its offset;
//  2. every edge finds its position in U_g by binary search and sets its bit
//     with atomicOr in the tile mask (bit order is exact, so the masks are
//     deterministic whatever the atomic order);
//  3. tile popcounts decide kept tiles; listed blocks are compacted with a
//     scan in ascending (group, block) order;
//  4. the residual CSR is one exclusive scan over the per-edge flags "tile not
//     kept" (edges stay in CSR order, so columns stay ascending).
// Count-sorted packing (packing GNN_PACK_COUNT) orders each group's columns
// by descending number of edges in the group, ties by ascending id, before
// cutting them into blocks: the run length of each (group, source) key in the
// sorted key list is its count, and one more radix sort of (group, 255 -
// count, source) keys gives the packed order; every edge then maps its
// id-sorted position to its packed position.
// Planning runs the same pass without writing the output and reads the
// counts back (synchronous).
#include <cub/device/device_radix_sort.cuh>
#include <cub/device/device_scan.cuh>

#include <algorithm>

#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);

namespace {

constexpr int kGroupRows = 128;

int bits_of(int64_t v) {
    int b = 1;
    while (b < 63 && ((int64_t)1 << b) <= v) ++b;
    return b;
}

int nblocks(int64_t n, int t = 256) { return (int)std::max<int64_t>(1, (n + t - 1) / t); }

// row of every edge (one warp per row)
__global__ void k_bs_rows(const int32_t *__restrict__ rowptr, int32_t n, int32_t *__restrict__ rowid) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= n) return;
    for (int32_t k = rowptr[r] + lane; k < rowptr[r + 1]; k += 32) rowid[k] = (int32_t)r;
}

__global__ void k_bs_keys(const int32_t *__restrict__ rowid, const int32_t *__restrict__ colidx, int64_t m,
                          uint64_t *__restrict__ key) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < m; e += stride)
        key[e] = ((uint64_t)(uint32_t)(rowid[e] / kGroupRows) << 32) | (uint32_t)colidx[e];
}

// first occurrence of each (group, source) key; per-group unique counts
__global__ void k_bs_unique(const uint64_t *__restrict__ key, int64_t m, int32_t *__restrict__ uflag,
                            int32_t *__restrict__ nu) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < m; k += stride) {
        const bool first = k == 0 || key[k] != key[k - 1];
        uflag[k] = first ? 1 : 0;
        if (first) atomicAdd(&nu[(int32_t)(key[k] >> 32)], 1);
    }
}

// U[u] = source of the u-th unique key; first (may be null) = position of
// its first occurrence in the sorted keys, and first[n_unique] = m
__global__ void k_bs_ulist(const uint64_t *__restrict__ key, const int32_t *__restrict__ uflag,
                           const int32_t *__restrict__ upos, int64_t m, int32_t *__restrict__ U,
                           int32_t *__restrict__ first) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < m; k += stride) {
        if (uflag[k]) {
            U[upos[k]] = (int32_t)(uint32_t)key[k];
            if (first) first[upos[k]] = (int32_t)k;
        }
        if (first && k == m - 1) first[upos[k] + uflag[k]] = (int32_t)m;
    }
}

// packing keys of the unique (group, source) pairs: (group, 255 - count,
// source), whose ascending order is the group's columns by descending edge
// count, ties by ascending id (a count is at most the group's 128 rows)
__global__ void k_bs_pack_keys(const uint64_t *__restrict__ key, const int32_t *__restrict__ first,
                               int64_t nuniq, uint64_t *__restrict__ pk, int32_t *__restrict__ pv) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nuniq; u += stride) {
        const uint64_t k = key[first[u]];
        const uint64_t cnt = (uint64_t)(first[u + 1] - first[u]);
        pk[u] = ((k >> 32) << 40) | ((255ull - cnt) << 32) | (k & 0xffffffffull);
        pv[u] = (int32_t)u;
    }
}

// rank[u] = packed position of unique u (in the same group-major numbering);
// P[q] = the source at packed position q (P may alias pv: thread q reads
// pv[q] before it writes P[q])
__global__ void k_bs_pack_rank(const uint64_t *__restrict__ pk, const int32_t *pv, int64_t nuniq,
                               int32_t *__restrict__ rank, int32_t *P) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < nuniq; q += stride) {
        const int32_t u = pv[q];
        rank[u] = (int32_t)q;
        P[q] = (int32_t)(uint32_t)pk[q];
    }
}

__global__ void k_bs_nblk(const int32_t *__restrict__ nu, int32_t ng, int32_t *__restrict__ nblk) {
    const int32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g < ng) nblk[g] = (nu[g] + 15) / 16;
    if (g == ng) nblk[g] = 0;
}

// set each edge's bit in its tile mask; remember its tile
__global__ void k_bs_place(const int32_t *__restrict__ rowid, const int32_t *__restrict__ colidx, int64_t m,
                           const int32_t *__restrict__ U, const int32_t *__restrict__ uoff,
                           const int32_t *__restrict__ nu, const int32_t *__restrict__ boff,
                           const int32_t *__restrict__ rank, unsigned long long *__restrict__ mask,
                           int32_t *__restrict__ tile_of) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < m; e += stride) {
        const int32_t i = rowid[e], j = colidx[e], g = i / kGroupRows;
        const int32_t *u = U + uoff[g];
        int32_t lo = 0, hi = nu[g] - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if (u[mid] < j) lo = mid + 1; else hi = mid;
        }
        // packed position (count-sorted packing); the id order otherwise
        if (rank) lo = rank[uoff[g] + lo] - uoff[g];
        const int32_t b = lo / 16, c = lo % 16, w = (i % kGroupRows) / 16, r = i % 16;
        const int32_t bit = r * 16 + c;
        const int64_t t = ((int64_t)boff[g] + b) * 8 + w;
        atomicOr(mask + t * 4 + bit / 64, 1ull << (bit % 64));
        tile_of[e] = (int32_t)t;
    }
}

// kept[t], listed[block]; counts[1] += kept tiles, counts[2] += their edges
__global__ void k_bs_tiles(const unsigned long long *__restrict__ mask, int64_t nt, float thr,
                           uint8_t *__restrict__ kept, int32_t *__restrict__ listed,
                           unsigned long long *__restrict__ counts) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < nt; t += stride) {
        int p = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) p += __popcll(mask[t * 4 + q]);
        const bool k = p >= 1 && ((float)p / 256.0f >= thr);
        kept[t] = k ? 1 : 0;
        if (k) {
            listed[t / 8] = 1;
            atomicAdd(&counts[1], 1ull);
            atomicAdd(&counts[2], (unsigned long long)p);
        }
    }
}

__global__ void k_bs_block_group(const int32_t *__restrict__ boff, int32_t ng, int32_t *__restrict__ bgrp) {
    const int32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= ng) return;
    for (int32_t b = boff[g]; b < boff[g + 1]; ++b) bgrp[b] = g;
}

// write listed blocks: columns and masks (zero for tiles not kept)
__global__ void k_bs_emit(const int32_t *__restrict__ listed, const int32_t *__restrict__ lpos, int64_t nb,
                          const int32_t *__restrict__ bgrp, const int32_t *__restrict__ boff,
                          const int32_t *__restrict__ uoff, const int32_t *__restrict__ nu,
                          const int32_t *__restrict__ cols_of, const unsigned long long *__restrict__ mask,
                          const uint8_t *__restrict__ kept, int32_t *__restrict__ blk_cols,
                          unsigned long long *__restrict__ blk_mask) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t bk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; bk < nb; bk += stride) {
        if (!listed[bk]) continue;
        const int64_t o = lpos[bk];
        const int32_t g = bgrp[bk], b = (int32_t)(bk - boff[g]);
        for (int c = 0; c < 16; ++c) {
            const int32_t p = 16 * b + c;
            blk_cols[o * 16 + c] = p < nu[g] ? cols_of[uoff[g] + p] : 0;
        }
        for (int w = 0; w < 8; ++w)
            for (int q = 0; q < 4; ++q)
                blk_mask[(o * 8 + w) * 4 + q] = kept[bk * 8 + w] ? mask[(bk * 8 + w) * 4 + q] : 0ull;
    }
}

__global__ void k_bs_grp_offsets(const int32_t *__restrict__ boff, const int32_t *__restrict__ lpos, int32_t ng,
                                 int32_t *__restrict__ out) {
    const int32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    if (g <= ng) out[g] = lpos[boff[g]];
}

__global__ void k_bs_resflag(const int32_t *__restrict__ tile_of, const uint8_t *__restrict__ kept, int64_t m,
                             int32_t *__restrict__ rflag) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < m; e += stride)
        rflag[e] = kept[tile_of[e]] ? 0 : 1;
    if (blockIdx.x == 0 && threadIdx.x == 0) rflag[m] = 0;
}

__global__ void k_bs_residual(const int32_t *__restrict__ colidx, const int32_t *__restrict__ rflag,
                              const int32_t *__restrict__ rpos, int64_t m, int32_t *__restrict__ res_colidx) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < m; e += stride)
        if (rflag[e]) res_colidx[rpos[e]] = colidx[e];
}

__global__ void k_bs_res_rowptr(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ rpos, int32_t n,
                                int32_t *__restrict__ res_rowptr) {
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i <= n) res_rowptr[i] = rpos[rowptr[i]];
}

struct BsWs {
    int32_t *rowid, *uflag, *upos, *U, *tile_of, *rflag, *rpos;
    uint64_t *key[2];
    int32_t *nu, *uoff, *nblk, *boff;
    unsigned long long *mask;  // [max blocks * 8 tiles * 4 words]
    uint8_t *kept;             // [max blocks * 8]
    int32_t *listed, *lpos, *bgrp;
    unsigned long long *counts;  // [0] listed blocks, [1] kept tiles, [2] tile edges
    void *temp;
    size_t temp_bytes;
    int64_t max_blocks;
    size_t bytes;
};

BsWs bs_layout(const gnn_csr *g, void *base) {
    Carver c(base);
    BsWs W;
    const int64_t m = g->nnz;
    const int32_t ng = (g->n_rows + kGroupRows - 1) / kGroupRows;
    W.max_blocks = m / 16 + ng + 1;
    W.rowid = c.take<int32_t>(m);
    W.uflag = c.take<int32_t>(m + 1);
    W.upos = c.take<int32_t>(m + 1);
    W.U = c.take<int32_t>(m);
    W.tile_of = c.take<int32_t>(m);
    W.rflag = c.take<int32_t>(m + 1);
    W.rpos = c.take<int32_t>(m + 1);
    W.key[0] = c.take<uint64_t>(m);
    W.key[1] = c.take<uint64_t>(m);
    W.nu = c.take<int32_t>(ng + 1);
    W.uoff = c.take<int32_t>(ng + 1);
    W.nblk = c.take<int32_t>(ng + 1);
    W.boff = c.take<int32_t>(ng + 1);
    W.mask = c.take<unsigned long long>((size_t)W.max_blocks * 32);
    W.kept = c.take<uint8_t>((size_t)W.max_blocks * 8);
    W.listed = c.take<int32_t>(W.max_blocks + 1);
    W.lpos = c.take<int32_t>(W.max_blocks + 1);
    W.bgrp = c.take<int32_t>(W.max_blocks);
    W.counts = c.take<unsigned long long>(4);
    size_t t = 0, x = 0;
    cub::DeviceRadixSort::SortKeys(nullptr, x, (const uint64_t *)nullptr, (uint64_t *)nullptr, m);
    t = std::max(t, x);
    cub::DeviceRadixSort::SortPairs(nullptr, x, (const uint64_t *)nullptr, (uint64_t *)nullptr,
                                    (const int32_t *)nullptr, (int32_t *)nullptr, m);
    t = std::max(t, x);
    cub::DeviceScan::ExclusiveSum(nullptr, x, (const int32_t *)nullptr, (int32_t *)nullptr,
                                  std::max<int64_t>(m + 1, W.max_blocks + 1));
    t = std::max(t, x);
    W.temp_bytes = t;
    W.temp = c.take<char>(t);
    W.bytes = c.used;
    return W;
}

struct BsOut {
    int32_t *grp_blk_offset, *blk_cols, *res_rowptr, *res_colidx;
    uint64_t *blk_mask;
    size_t bytes;
};

BsOut bs_out_layout(int32_t n_rows, int64_t n_blocks, int64_t nnz_res, void *base) {
    Carver c(base);
    BsOut o;
    const int32_t ng = (n_rows + kGroupRows - 1) / kGroupRows;
    o.grp_blk_offset = c.take<int32_t>(ng + 1);
    o.blk_cols = c.take<int32_t>((size_t)n_blocks * 16);
    o.blk_mask = c.take<uint64_t>((size_t)n_blocks * 32);
    o.res_rowptr = c.take<int32_t>((size_t)n_rows + 1);
    o.res_colidx = c.take<int32_t>((size_t)std::max<int64_t>(nnz_res, 1));
    o.bytes = c.used;
    return o;
}

#define GNN_TRY(x)                                                \
    do {                                                          \
        cudaError_t e__ = (x);                                    \
        if (e__ != cudaSuccess) return ::gnn::cuda_status(e__);   \
    } while (0)

// The whole pass (synchronous).  counts (host): {n_blocks, n_tiles_kept,
// nnz_tiles, nnz_residual}.  The layout is written only if out != nullptr,
// and then only if the counts equal `expect` (the plan the caller sized
// `out` with); otherwise GNN_ERR_INVALID_ARG and nothing is written.
gnn_status bs_pass(const gnn_csr *g, float thr, int32_t packing, BsWs &W, const BsOut *out,
                   const int64_t *expect, int64_t *counts, cudaStream_t s) {
    // count-sorted packing reuses scratch that is free at that point: the
    // unsorted keys and the unique flags / positions (read only by k_bs_ulist)
    // hold the packing keys and values, and the residual flags / positions
    // (written only after k_bs_place) hold the first occurrences and ranks
    const bool pack = packing == GNN_PACK_COUNT;
    int32_t *first = pack ? W.rflag : nullptr;
    int32_t *rank = pack ? W.rpos : nullptr;
    int32_t *packed_cols = pack ? W.upos : nullptr;
    const int32_t n = g->n_rows;
    const int64_t m = g->nnz;
    const int32_t ng = (n + kGroupRows - 1) / kGroupRows;
    size_t tb = W.temp_bytes;
    const int gs = std::min(nblocks(m), sm_count() * 8);
    GNN_TRY(cudaMemsetAsync(W.nu, 0, sizeof(int32_t) * (ng + 1), s));
    GNN_TRY(cudaMemsetAsync(W.counts, 0, sizeof(unsigned long long) * 4, s));
    if (m > 0) {
        k_bs_rows<<<nblocks((int64_t)n * 32), 256, 0, s>>>(g->rowptr, n, W.rowid);
        k_bs_keys<<<gs, 256, 0, s>>>(W.rowid, g->colidx, m, W.key[0]);
        note_launch(2);
        GNN_TRY(cub::DeviceRadixSort::SortKeys(W.temp, tb, W.key[0], W.key[1], m, 0, 32 + bits_of(ng), s));
        k_bs_unique<<<gs, 256, 0, s>>>(W.key[1], m, W.uflag, W.nu);
        note_launch(2);
        GNN_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.uflag, W.upos, m, s));
        k_bs_ulist<<<gs, 256, 0, s>>>(W.key[1], W.uflag, W.upos, m, W.U, first);
        note_launch(2);
        if (pack) {
            int32_t last_pos = 0, last_flag = 0;
            GNN_TRY(cudaMemcpyAsync(&last_pos, W.upos + m - 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
            GNN_TRY(cudaMemcpyAsync(&last_flag, W.uflag + m - 1, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
            GNN_TRY(cudaStreamSynchronize(s));
            const int64_t nuniq = (int64_t)last_pos + last_flag;
            const int gu = std::min(nblocks(nuniq), sm_count() * 8);
            k_bs_pack_keys<<<gu, 256, 0, s>>>(W.key[1], first, nuniq, W.key[0], W.uflag);
            note_launch();
            // sorted packing keys into key[1] (the sorted edge keys are no
            // longer needed), their unique ids into upos
            GNN_TRY(cub::DeviceRadixSort::SortPairs(W.temp, tb, W.key[0], W.key[1], W.uflag, W.upos, nuniq,
                                                    0, 40 + bits_of(ng), s));
            k_bs_pack_rank<<<gu, 256, 0, s>>>(W.key[1], W.upos, nuniq, rank, packed_cols);
            note_launch(2);
        }
    }
    GNN_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.nu, W.uoff, ng + 1, s));
    k_bs_nblk<<<nblocks(ng + 1), 256, 0, s>>>(W.nu, ng, W.nblk);
    note_launch(2);
    GNN_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.nblk, W.boff, ng + 1, s));
    note_launch();
    int32_t total_blocks = 0;
    GNN_TRY(cudaMemcpyAsync(&total_blocks, W.boff + ng, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_TRY(cudaStreamSynchronize(s));
    if (total_blocks > W.max_blocks) return GNN_ERR_DEVICE_CHECK;
    const int64_t nt = (int64_t)total_blocks * 8;
    GNN_TRY(cudaMemsetAsync(W.mask, 0, sizeof(unsigned long long) * (size_t)nt * 4, s));
    GNN_TRY(cudaMemsetAsync(W.listed, 0, sizeof(int32_t) * ((size_t)total_blocks + 1), s));
    if (m > 0) {
        k_bs_place<<<gs, 256, 0, s>>>(W.rowid, g->colidx, m, W.U, W.uoff, W.nu, W.boff, rank, W.mask,
                                      W.tile_of);
        note_launch();
    }
    if (nt > 0) {
        k_bs_tiles<<<std::min(nblocks(nt), sm_count() * 8), 256, 0, s>>>(W.mask, nt, thr, W.kept, W.listed,
                                                                            W.counts);
        note_launch();
    }
    GNN_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.listed, W.lpos, total_blocks + 1, s));
    note_launch();
    // residual flags and positions
    if (m > 0) {
        k_bs_resflag<<<gs, 256, 0, s>>>(W.tile_of, W.kept, m, W.rflag);
        note_launch();
    } else {
        GNN_TRY(cudaMemsetAsync(W.rflag, 0, sizeof(int32_t), s));
    }
    GNN_TRY(cub::DeviceScan::ExclusiveSum(W.temp, tb, W.rflag, W.rpos, m + 1, s));
    note_launch();
    int32_t listed_total = 0, res_total = 0;
    GNN_TRY(cudaMemcpyAsync(&listed_total, W.lpos + total_blocks, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_TRY(cudaMemcpyAsync(&res_total, W.rpos + m, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    unsigned long long hc[4] = {0, 0, 0, 0};
    GNN_TRY(cudaMemcpyAsync(hc, W.counts, sizeof(hc), cudaMemcpyDeviceToHost, s));
    GNN_TRY(cudaStreamSynchronize(s));
    counts[0] = listed_total;
    counts[1] = (int64_t)hc[1];
    counts[2] = (int64_t)hc[2];
    counts[3] = res_total;
    if (!out) return GNN_OK;
    if (!expect || expect[0] != counts[0] || expect[3] != counts[3]) return GNN_ERR_INVALID_ARG;
    k_bs_block_group<<<nblocks(ng), 256, 0, s>>>(W.boff, ng, W.bgrp);
    note_launch();
    if (total_blocks > 0) {
        k_bs_emit<<<std::min(nblocks(total_blocks), sm_count() * 8), 256, 0, s>>>(
            W.listed, W.lpos, total_blocks, W.bgrp, W.boff, W.uoff, W.nu, pack ? packed_cols : W.U, W.mask,
            W.kept, out->blk_cols,
            reinterpret_cast<unsigned long long *>(out->blk_mask));
        note_launch();
    }
    k_bs_grp_offsets<<<nblocks(ng + 1), 256, 0, s>>>(W.boff, W.lpos, ng, out->grp_blk_offset);
    k_bs_res_rowptr<<<nblocks((int64_t)n + 1), 256, 0, s>>>(g->rowptr, W.rpos, n, out->res_rowptr);
    note_launch(2);
    if (m > 0 && res_total > 0) {
        k_bs_residual<<<gs, 256, 0, s>>>(g->colidx, W.rflag, W.rpos, m, out->res_colidx);
        note_launch();
    }
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

}  // namespace

size_t blocksparse_workspace_bytes(const gnn_csr *g) { return bs_layout(g, nullptr).bytes; }

}  // namespace gnn

using namespace gnn;

extern "C" {

gnn_status gnn_blocksparse_plan_packed(const gnn_csr *g, float fill_threshold, int32_t packing, void *ws,
                                       size_t ws_bytes, gnn_blocksparse *bs, size_t *out_bytes,
                                       void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!bs || !out_bytes) return GNN_ERR_INVALID_ARG;
    if (!(fill_threshold >= 0.f && fill_threshold <= 1.f)) return GNN_ERR_INVALID_ARG;
    if (packing != GNN_PACK_ID && packing != GNN_PACK_COUNT) return GNN_ERR_INVALID_ARG;
    BsWs W = bs_layout(g, ws);
    if (!ws || ws_bytes < W.bytes) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    int64_t c[4] = {0, 0, 0, 0};
    st = bs_pass(g, fill_threshold, packing, W, nullptr, nullptr, c, as_stream(stream));
    if (st != GNN_OK) return st;
    *bs = gnn_blocksparse{};
    bs->packing = packing;
    bs->n_rows = g->n_rows;
    bs->n_groups = (g->n_rows + kGroupRows - 1) / kGroupRows;
    bs->n_blocks = c[0];
    bs->n_tiles_kept = c[1];
    bs->nnz_tiles = c[2];
    bs->nnz_residual = c[3];
    bs->fill_threshold = fill_threshold;
    *out_bytes = bs_out_layout(g->n_rows, c[0], c[3], nullptr).bytes;
    return GNN_OK;
}

gnn_status gnn_blocksparse_plan(const gnn_csr *g, float fill_threshold, void *ws, size_t ws_bytes,
                                gnn_blocksparse *bs, size_t *out_bytes, void *stream) {
    return gnn_blocksparse_plan_packed(g, fill_threshold, GNN_PACK_ID, ws, ws_bytes, bs, out_bytes, stream);
}

gnn_status gnn_blocksparse_build(const gnn_csr *g, gnn_blocksparse *bs, void *out, size_t out_bytes, void *ws,
                                 size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!bs || !out || bs->n_rows != g->n_rows) return GNN_ERR_INVALID_ARG;
    if (bs->packing != GNN_PACK_ID && bs->packing != GNN_PACK_COUNT) return GNN_ERR_INVALID_ARG;
    if (!aligned256(out) || !aligned256(ws)) return GNN_ERR_INVALID_ARG;
    BsOut o = bs_out_layout(g->n_rows, bs->n_blocks, bs->nnz_residual, out);
    if (out_bytes < o.bytes) return GNN_ERR_WORKSPACE;
    BsWs W = bs_layout(g, ws);
    if (!ws || ws_bytes < W.bytes) return GNN_ERR_WORKSPACE;
    int64_t c[4];
    const int64_t expect[4] = {bs->n_blocks, bs->n_tiles_kept, bs->nnz_tiles, bs->nnz_residual};
    st = bs_pass(g, bs->fill_threshold, bs->packing, W, &o, expect, c, as_stream(stream));
    if (st != GNN_OK) return st;
    bs->grp_blk_offset = o.grp_blk_offset;
    bs->blk_cols = o.blk_cols;
    bs->blk_mask = o.blk_mask;
    bs->res_rowptr = o.res_rowptr;
    bs->res_colidx = o.res_colidx;
    return GNN_OK;
}

}  // extern "C"
