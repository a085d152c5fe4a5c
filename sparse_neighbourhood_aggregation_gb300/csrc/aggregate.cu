// Steps a1 (SpMM) and a2 (segment sum / mean / max) of CSR neighbourhood
// aggregation.
//
// IO-aware GNN layers, Section 2.2 (i)-(ii), Section 3.1 and Appendix D.1
// ("degree-aware reduction", light/heavy split, packed (value, index)
// merge), Section 4.1 / Appendix E.1 (feature- vs neighbour-parallel
// mappings).
//
// GB300 design.  All three families stream 16-byte feature chunks with
// 128-bit loads; rows are 16-byte aligned.  Two AUTO schedules split the
// edge list, instead of one block per node, so every warp does about the
// same number of loads:
//  - k_agg_span (rows of 32 chunks, prepared graph given): spans of 64 edges
//    from the prepared graph, light rows kept whole, heavy rows cut, row
//    closes read from prepared row-end bits; heavy-row pieces are stored
//    with plain stores (max: folded by 64-bit max reductions) and finalised,
//    in edge order, by k_agg_span_fix.
//  - k_agg_auto (any width, with or without the prepared graph): runs of E
//    edges per group of LPR lanes (a "worker"); light rows packed several to
//    a worker, heavy rows split across ceil(deg/E) workers; a row that
//    crosses a run boundary leaves one partial result per worker, folded by
//    atomics into the slot of its first run, and the last worker to arrive
//    (a ticket counter, no spinning) finalises it.
// Loads of U consecutive edges are issued before any of them is accumulated,
// whatever row they belong to, which keeps U 16-byte loads in flight per lane
// even through runs of degree-1 rows.  Sums of a row cut into three or more
// pieces are fp32-order dependent in k_agg_auto (the pieces arrive in any
// order; k_agg_span adds them in edge order); max
// merges (value, source id) pairs under the order-preserving key with ties
// to the smaller id -- the paper's packed 64-bit atomic merge -- and is
// exact and deterministic.
#include <algorithm>
#include <mutex>

#include "async.cuh"
#include "common.cuh"

// Minimum resident 256-thread blocks per SM requested for the one-chunk-per-
// lane AUTO kernels (register cap 65536 / (256 * GNN_AGG_MINB)).
#ifndef GNN_AGG_MINB
#define GNN_AGG_MINB 4
#endif
// AUTO runs are GNN_AGG_RUNMUL runs of the prepared graph's run table
// (kRunEdges edges each): longer runs amortise each worker's start-up chain
// of dependent loads (run table -> row pointers -> column ids -> rows)
#ifndef GNN_AGG_RUNMUL
#define GNN_AGG_RUNMUL 1
#endif
// 16-byte loads in flight per lane in the edge loops
#ifndef GNN_AGG_U
#define GNN_AGG_U 4
#endif

namespace gnn {

void prep_pointers(const gnn_csr *g, const void *prep, const int32_t **d_out,
                   const float **dinv_in, const float **dinv_out);
gnn_status check_csr_args(const gnn_csr *g);
const int32_t *prep_run_table(const gnn_csr *g, const void *prep);
void prep_span_tables(const gnn_csr *g, const void *prep, const uint32_t **win_flags,
                      const int32_t **win_rowbase, const int32_t **ne_rows,
                      const int32_t **sp_begin, const int4 **items, const int32_t **items_count,
                      const int32_t **win_rowstart);

enum AggOp { AGG_WSUM = 0, AGG_MEAN = 1, AGG_MAX = 2, AGG_MIN = 3 };
// max and min share one code path: min keeps the complement of the order
// key, so the largest stored key is the smallest value, and every packed
// (key << 32) | ~source_id merge by unsigned maximum serves both (ties to
// the smaller id).
__host__ __device__ constexpr bool is_ext(int op) { return op == AGG_MAX || op == AGG_MIN; }
// per-edge weight source / per-row factor source
enum ColMode { COL_ONE = 0, COL_RSQRT = 1, COL_RECIP = 2 };
enum RowMode { ROW_ONE = 0, ROW_RSQRT = 1, ROW_RECIP = 2 };

struct AggArgs {
    const int32_t *rowptr;
    const int32_t *colidx;
    const float *values;    // per-edge values or null
    const int32_t *d_out;   // for COL_RECIP
    const float *dinv_in;   // for ROW_RSQRT
    const float *dinv_out;  // for COL_RSQRT
    const uint4 *X;         // [n_cols, V] 16-byte chunks
    float *Y;
    int32_t *argmax;
    float *carry;           // [n_workers, F] fp32 (max: [n_workers, F] uint64)
    int32_t *tickets;       // [n_workers], zero on entry and on exit
    const int32_t *run_first_row;  // [n_workers+1] from the prepared graph, or null
    const uint32_t *win_flags;     // prepared row-end bits, one word per 32 edges
    const int32_t *win_rowbase;    // prepared rank of the row holding edge 32*win
    const int32_t *ne_rows;        // prepared non-empty rows, ascending
    const int32_t *sp_begin;       // prepared first edge of each edge span
    const int32_t *win_rowstart;   // prepared first edge of the row holding edge 32*win
    const int4 *items;             // prepared heavy-row chunks {row, begin, end, chunk}
    const int32_t *items_count;    // prepared number of items
    int32_t n_spans;               // edge-span kernel: spans of 1 << span_shift edges
    int32_t span_shift;
    int64_t nnz;
    int64_t n_workers;
    int32_t n_rows;
    int32_t F;              // features
    int32_t V;              // 16-byte chunks per row
    int32_t lpr;            // lanes per worker (8, 16 or 32)
    int32_t E;              // edges per worker (multiple of 32)
    int32_t col_mode, row_mode;
};

template <int OP, class T, int CPL>
struct Acc {
    static constexpr int NV = Chunk<T>::N;
    static constexpr bool MX = is_ext(OP);
    float v[MX ? 1 : CPL][MX ? 1 : NV];      // sums
    uint32_t km[MX ? CPL : 1][MX ? NV : 1];  // max: order_key of the maximum (min: its complement), 0 = none
    int32_t idx[MX ? CPL : 1][MX ? NV : 1];  // its source id, -1 = nothing seen

    // every finite value's key is > 0, so a key of 0 means "no edge yet"
    __device__ __forceinline__ uint32_t key(int c, int k) const { return km[c][k]; }
    __device__ __forceinline__ float max_value(int c, int k) const {
        return km[c][k] ? key_value(OP == AGG_MIN ? ~km[c][k] : km[c][k]) : 0.f;
    }
    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                if (MX) { km[c][k] = 0u; idx[c][k] = -1; }
                else v[c][k] = 0.f;
            }
    }
    __device__ __forceinline__ void add(const uint4 *x, float w, int32_t j) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            float f[NV];
            Chunk<T>::unpack(x[c], f);
            if (MX) {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const uint32_t kk = OP == AGG_MIN ? ~order_key(f[k]) : order_key(f[k]);
                    // edges arrive in ascending source id: strict > keeps the
                    // smallest id among equal keys
                    if (kk > km[c][k]) { km[c][k] = kk; idx[c][k] = j; }
                }
            } else {
                // v += w * f on pairs of features (one rounding each, as fmaf)
                const uint64_t ww = pk2(w, w);
#pragma unroll
                for (int k = 0; k < NV; k += 2)
                    upk2(fma2(ww, pk2(f[k], f[k + 1]), pk2(v[c][k], v[c][k + 1])), v[c][k], v[c][k + 1]);
            }
        }
    }
    // merged state from a packed (key << 32) | ~id word
    __device__ __forceinline__ void set_packed(int c, int k, unsigned long long p) {
        km[c][k] = (uint32_t)(p >> 32);
        idx[c][k] = (int32_t)(0xFFFFFFFFu - (uint32_t)p);
    }
};

__device__ __forceinline__ float row_factor(const AggArgs &a, int32_t r, int32_t deg) {
    if (a.row_mode == ROW_RSQRT) return a.dinv_in[r];
    if (a.row_mode == ROW_RECIP) return deg > 0 ? __frcp_rn((float)deg) : 0.f;
    return 1.f;
}

__device__ __forceinline__ float edge_weight(const AggArgs &a, int64_t e, int32_t j) {
    float w = a.values ? __ldg(a.values + e) : 1.f;
    if (a.col_mode == COL_RSQRT) w *= __ldg(a.dinv_out + j);
    else if (a.col_mode == COL_RECIP) w *= __frcp_rn((float)__ldg(a.d_out + j));
    return w;
}

// Output rows are written once and never read by the kernel: streaming
// stores (st.global.cs, evict-first) keep them from displacing gathered
// feature rows in L2.
#ifndef GNN_Y_STREAM
#define GNN_Y_STREAM 1
#endif
// Column ids are read once: streaming loads (ld.global.cs).
#ifndef GNN_IDX_STREAM
#define GNN_IDX_STREAM 1
#endif

__device__ __forceinline__ void st_out4(float *p, float4 v) {
#if GNN_Y_STREAM
    __stcs(reinterpret_cast<float4 *>(p), v);
#else
    *reinterpret_cast<float4 *>(p) = v;
#endif
}
__device__ __forceinline__ void st_out4i(int32_t *p, int4 v) {
#if GNN_Y_STREAM
    __stcs(reinterpret_cast<int4 *>(p), v);
#else
    *reinterpret_cast<int4 *>(p) = v;
#endif
}
__device__ __forceinline__ int32_t ld_col(const int32_t *p) {
#if GNN_IDX_STREAM
    return __ldcs(p);
#else
    return __ldg(p);
#endif
}

// Store a finished row (fp32 features; the lane owns chunks c*lpr + gl).
template <int OP, class T, int CPL>
__device__ __forceinline__ void store_row(const AggArgs &a, int32_t r, int32_t deg,
                                          const Acc<OP, T, CPL> &acc, int gl) {
    constexpr int NV = Chunk<T>::N;
    float s = 1.f;
    if (OP == AGG_WSUM) s = row_factor(a, r, deg);
    const float inv_deg = (OP == AGG_MEAN && deg > 0) ? __frcp_rn((float)deg) : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        int64_t base = (int64_t)r * a.F + (int64_t)(c * a.lpr + gl) * NV;
        float o[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (OP == AGG_WSUM) o[k] = acc.v[c][k] * s;
            else if (OP == AGG_MEAN) o[k] = acc.v[c][k] * inv_deg;
            else o[k] = acc.max_value(c, k);
        }
#pragma unroll
        for (int k = 0; k < NV; k += 4) st_out4(a.Y + base + k, make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]));
        if (is_ext(OP) && a.argmax) {
#pragma unroll
            for (int k = 0; k < NV; k += 4)
                st_out4i(a.argmax + base + k,
                         make_int4(acc.idx[c][k], acc.idx[c][k + 1], acc.idx[c][k + 2], acc.idx[c][k + 3]));
        }
    }
}

template <int OP, class T, int CPL>
__device__ __forceinline__ void store_row_f(const AggArgs &a, int32_t r, int32_t deg, float rf,
                                            const Acc<OP, T, CPL> &acc, int gl) {
    constexpr int NV = Chunk<T>::N;
    float s = 1.f;
    if (OP == AGG_WSUM)
        s = a.row_mode == ROW_RSQRT ? rf : (a.row_mode == ROW_RECIP ? (deg > 0 ? __frcp_rn((float)deg) : 0.f) : 1.f);
    // mean: one correctly rounded reciprocal per row, then a product per feature
    const float inv_deg = (OP == AGG_MEAN && deg > 0) ? __frcp_rn((float)deg) : 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        int64_t base = (int64_t)r * a.F + (int64_t)(c * a.lpr + gl) * NV;
        float o[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (OP == AGG_WSUM) o[k] = acc.v[c][k] * s;
            else if (OP == AGG_MEAN) o[k] = acc.v[c][k] * inv_deg;
            else o[k] = acc.max_value(c, k);
        }
#pragma unroll
        for (int k = 0; k < NV; k += 4) st_out4(a.Y + base + k, make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]));
        if (is_ext(OP) && a.argmax) {
#pragma unroll
            for (int k = 0; k < NV; k += 4)
                st_out4i(a.argmax + base + k,
                         make_int4(acc.idx[c][k], acc.idx[c][k + 1], acc.idx[c][k + 2], acc.idx[c][k + 3]));
        }
    }
}

// Partial row of a heavy row r (degree > E).  Every run that holds a piece of
// r folds it into the row's accumulation slot -- slot wa, the run the row
// starts in -- with vector fp32 atomics (sum-like ops) or, for max, with a
// 64-bit atomicMax on (key << 32) | ~source_id, the packed (value, index)
// merge of IO-aware GNN layers, Appendix D.1 (ties resolve to the smallest
// id).  A ticket counter per slot tells the last piece to arrive, which
// finalises the row and leaves the slot and ticket at zero again.
template <int OP, class T, int CPL>
__device__ __forceinline__ void flush_partial(const AggArgs &a, int64_t w, int slot, int32_t r,
                                              Acc<OP, T, CPL> &acc, int gl, unsigned gmask) {
    (void)w;
    (void)slot;
    constexpr int NV = Chunk<T>::N;
    const int64_t F = a.F;
    const int32_t rb = __ldg(a.rowptr + r), re = __ldg(a.rowptr + r + 1);
    const int64_t wa = (int64_t)rb / a.E, wb = ((int64_t)re - 1) / a.E;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int64_t off = wa * F + (int64_t)(c * a.lpr + gl) * NV;
#pragma unroll
        for (int k = 0; k < NV; k += 4) {
            if (is_ext(OP)) {
                unsigned long long *dst = reinterpret_cast<unsigned long long *>(a.carry) + off + k;
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    const uint32_t key = acc.key(c, k + z);
                    const unsigned long long packed =
                        ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)acc.idx[c][k + z]);
                    atomicMax(dst + z, packed);
                }
            } else {
                atomicAdd(reinterpret_cast<float4 *>(a.carry + off + k),
                          make_float4(acc.v[c][k], acc.v[c][k + 1], acc.v[c][k + 2], acc.v[c][k + 3]));
            }
        }
    }
    __threadfence();
    __syncwarp(gmask);
    int t = 0;
    if (gl == 0) t = atomicAdd(a.tickets + wa, 1);
    t = __shfl_sync(gmask, t, 0, a.lpr);
    if (t != (int)(wb - wa)) return;
    __threadfence();
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int64_t off = wa * F + (int64_t)(c * a.lpr + gl) * NV;
#pragma unroll
        for (int k = 0; k < NV; k += 4) {
            if (is_ext(OP)) {
                unsigned long long *src = reinterpret_cast<unsigned long long *>(a.carry) + off + k;
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    acc.set_packed(c, k + z, __ldcg(src + z));
                    src[z] = 0ull;
                }
            } else {
                float4 *src = reinterpret_cast<float4 *>(a.carry + off + k);
                const float4 pv = __ldcg(src);
                acc.v[c][k] = pv.x;
                acc.v[c][k + 1] = pv.y;
                acc.v[c][k + 2] = pv.z;
                acc.v[c][k + 3] = pv.w;
                *src = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    store_row<OP, T, CPL>(a, r, re - rb, acc, gl);
    __syncwarp(gmask);
    if (gl == 0) a.tickets[wa] = 0;
}

// First row r with rowptr[r] >= e (rowptr[n_rows] >= e assumed), found by the
// lpr lanes of a group together: each round every lane probes one position
// of the current interval and a ballot narrows it by a factor of lpr.
__device__ __forceinline__ int32_t group_lower_bound(const int32_t *__restrict__ rowptr,
                                                     int32_t n_rows, int32_t e, int gl, int lpr,
                                                     unsigned gmask) {
    int32_t lo = 0, hi = n_rows;  // answer in [lo, hi]
    while (hi - lo > 1) {
        int32_t span = hi - lo;
        int32_t step = (span + lpr - 1) / lpr;
        int32_t pos = lo + gl * step;            // probe rowptr[pos] < e ?
        bool below = pos < hi && __ldg(rowptr + pos) < e;
        unsigned b = __ballot_sync(gmask, below);
        if (lpr < 32) b = (b >> ((threadIdx.x & 31) & ~(lpr - 1))) & ((1u << lpr) - 1u);
        int nb = __popc(b);                       // probes 0..nb-1 are below e
        if (nb == 0) { hi = lo; break; }
        int32_t new_lo = lo + (nb - 1) * step + 1;  // first index not known below
        int32_t new_hi = min(hi, lo + nb * step);
        lo = new_lo;
        hi = new_hi;
        if (lo >= hi) break;
    }
    // lo is the answer unless rowptr[lo] < e (possible when hi - lo == 1)
    if (lo < n_rows && __ldg(rowptr + lo) < e) ++lo;
    return lo;
}

// Accumulate the edges [b, end) of one row into acc (no row changes).
template <int OP, class T, int CPL>
__device__ __forceinline__ void run_segment(const AggArgs &a, int32_t b, int32_t end,
                                            Acc<OP, T, CPL> &acc, int gl, unsigned gmask,
                                            bool weighted) {
    constexpr int U = CPL >= GNN_AGG_U ? 1 : GNN_AGG_U / CPL;
    const int lpr = a.lpr;
    for (int32_t cb = b; cb < end; cb += lpr) {
        int32_t cj = (cb + gl < end) ? __ldg(a.colidx + cb + gl) : 0;
        float cw = (weighted && cb + gl < end) ? edge_weight(a, cb + gl, cj) : 1.f;
        const int n = min(lpr, end - cb);
        for (int u0 = 0; u0 < n; u0 += U) {
            uint4 xv[U][CPL];
            int32_t jv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                jv[u] = __shfl_sync(gmask, cj, u0 + u, lpr);
                if (u0 + u < n) {
                    const uint4 *src = a.X + (size_t)jv[u] * a.V + gl;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) xv[u][c] = ldg16(src + c * lpr);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float wt = weighted ? __shfl_sync(gmask, cw, u0 + u, lpr) : 1.f;
                if (u0 + u < n) acc.add(xv[u], wt, jv[u]);
            }
        }
    }
}

// AUTO mapping.  Run w covers edges [w*E, (w+1)*E).  A light row (degree
// <= E) belongs whole to the run its first edge falls in, so a run may read
// up to 2E-1 edges; a heavy row (degree > E) is cut at run boundaries and
// each run leaves a partial result that the row's last run merges.
template <int OP, class T, int CPL, int LPR>
__global__ void __launch_bounds__(256, (CPL <= 4 ? GNN_AGG_MINB : 2)) k_agg_auto(AggArgs a) {
    constexpr int U = CPL >= GNN_AGG_U ? 1 : GNN_AGG_U / CPL;
    // LPR > 0: lanes per worker known at compile time (32); 0: a.lpr
    const int lpr = LPR > 0 ? LPR : a.lpr;
    const int lane = threadIdx.x & 31;
    const int gl = lane & (lpr - 1);
    const unsigned gmask = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (lane & ~(lpr - 1)));
    const int32_t w = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / lpr);
    if (w >= a.n_workers) return;
    const int32_t nnz = (int32_t)a.nnz;
    const int32_t E = a.E;
    const int32_t e0 = w * E;
    const int32_t e1 = min(e0 + E, nnz);
    const int32_t *__restrict__ rowptr = a.rowptr;
    const int32_t n_rows = a.n_rows;
    const bool weighted = (OP == AGG_WSUM) && (a.values || a.col_mode != COL_ONE);

    // rows owned by this run: [lo, lo_end)
    int32_t lo, lo_end;
    if (a.run_first_row) {
        lo = __ldg(a.run_first_row + (int64_t)w * GNN_AGG_RUNMUL);
        lo_end = (w + 1 == a.n_workers) ? n_rows : __ldg(a.run_first_row + (int64_t)(w + 1) * GNN_AGG_RUNMUL);
    } else {
        lo = group_lower_bound(rowptr, n_rows, e0, gl, lpr, gmask);
        lo_end = (w + 1 == a.n_workers) ? n_rows : group_lower_bound(rowptr, n_rows, e1, gl, lpr, gmask);
    }

    Acc<OP, T, CPL> acc;
    acc.reset();

    // a heavy row that started in an earlier run and reaches into this one
    if (lo > 0 && e0 < nnz) {
        const int32_t lo_beg = __ldg(rowptr + lo);
        if (lo_beg > e0) {
            const int32_t h = lo - 1;
            const int32_t hb = __ldg(rowptr + h);
            if (lo_beg - hb > E) {
                run_segment<OP, T, CPL>(a, e0, min(lo_beg, e1), acc, gl, gmask, weighted);
                flush_partial<OP, T, CPL>(a, w, 0, h, acc, gl, gmask);
                acc.reset();
            }
        }
    }
    if (lo >= lo_end) return;

    // stream [s0, s1) over the owned rows lo .. rl
    const int32_t rl = lo_end - 1;
    const int32_t rl_beg = __ldg(rowptr + rl), rl_end = __ldg(rowptr + rl + 1);
    const bool heavy_tail = rl_end - rl_beg > E;
    const int32_t s0 = __ldg(rowptr + lo);
    const int32_t s1 = heavy_tail ? e1 : rl_end;

    // row-end (and row-factor) cache: lane k holds data of row rb + k
    int32_t r = lo, rb = lo;
    const bool rsq = OP == AGG_WSUM && a.row_mode == ROW_RSQRT;
    int32_t rp_cur = (rb + gl < n_rows) ? __ldg(rowptr + rb + gl + 1) : INT32_MAX;
    int32_t rp_nxt = (rb + lpr + gl < n_rows) ? __ldg(rowptr + rb + lpr + gl + 1) : INT32_MAX;
    float rf_cur = (rsq && rb + gl < n_rows) ? __ldg(a.dinv_in + rb + gl) : 1.f;
    float rf_nxt = (rsq && rb + lpr + gl < n_rows) ? __ldg(a.dinv_in + rb + lpr + gl) : 1.f;
    int32_t row_beg = s0;
    int32_t row_end = __shfl_sync(gmask, rp_cur, 0, lpr);

    auto finish_row = [&]() {
        float rf = __shfl_sync(gmask, rf_cur, r - rb, lpr);
        store_row_f<OP, T, CPL>(a, r, row_end - row_beg, rf, acc, gl);
        acc.reset();
    };
    auto advance = [&]() {
        ++r;
        if (r - rb == lpr) {
            rb = r;
            rp_cur = rp_nxt;
            rf_cur = rf_nxt;
            rp_nxt = (rb + lpr + gl < n_rows) ? __ldg(rowptr + rb + lpr + gl + 1) : INT32_MAX;
            if (rsq) rf_nxt = (rb + lpr + gl < n_rows) ? __ldg(a.dinv_in + rb + lpr + gl) : 1.f;
        }
        row_beg = row_end;
        row_end = __shfl_sync(gmask, rp_cur, r - rb, lpr);
    };

    // column / weight cache for edges [cb, cb+lpr); next window prefetched
    int32_t cb = s0;
    int32_t c_cur = (cb + gl < s1) ? __ldg(a.colidx + cb + gl) : 0;
    int32_t c_nxt = (cb + lpr + gl < s1) ? __ldg(a.colidx + cb + lpr + gl) : 0;
    float w_cur = 1.f, w_nxt = 1.f;
    if (weighted) {
        if (cb + gl < s1) w_cur = edge_weight(a, cb + gl, c_cur);
        if (cb + lpr + gl < s1) w_nxt = edge_weight(a, cb + lpr + gl, c_nxt);
    }
    const uint4 *__restrict__ X = a.X;
    const int32_t V = LPR > 0 ? LPR * CPL : a.V;
    for (int32_t eb = s0; eb < s1; eb += U) {
        if (eb - cb == lpr) {
            cb = eb;
            c_cur = c_nxt;
            w_cur = w_nxt;
            const int32_t en = cb + lpr + gl;
            c_nxt = en < s1 ? __ldg(a.colidx + en) : 0;
            if (weighted && en < s1) w_nxt = edge_weight(a, en, c_nxt);
        }
        uint4 xv[U][CPL];
        int32_t jv[U];
        const bool full = eb + U <= s1;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            jv[u] = __shfl_sync(gmask, c_cur, (eb - cb) + u, lpr);
            if (full || eb + u < s1) {
                const uint4 *src = X + (size_t)jv[u] * V + gl;
#pragma unroll
                for (int c = 0; c < CPL; ++c) xv[u][c] = ldg16(src + c * lpr);
            }
        }
        if (full && row_end >= eb + U) {
            // fast path: the whole batch lies inside the current row
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float wt = weighted ? __shfl_sync(gmask, w_cur, (eb - cb) + u, lpr) : 1.f;
                acc.add(xv[u], wt, jv[u]);
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t e = eb + u;
                if (e < s1) {
                    while (e == row_end) {
                        finish_row();
                        advance();
                    }
                    const float wt = weighted ? __shfl_sync(gmask, w_cur, (eb - cb) + u, lpr) : 1.f;
                    acc.add(xv[u], wt, jv[u]);
                }
            }
        }
    }
    // the row holding the last streamed edge, then empty rows up to rl
    if (r == rl && heavy_tail) {
        flush_partial<OP, T, CPL>(a, w, 1, r, acc, gl, gmask);
        return;
    }
    finish_row();
    while (r < rl) {
        advance();
        finish_row();
    }
}

// Edge-span AUTO kernel for rows of 32 16-byte chunks (fp32 F = 128, bf16
// F = 256), used when the prepared graph is given.  The prepared graph cuts
// the edge list into spans of about S = span_edges(nnz) edges: a row of degree
// <= S belongs whole to the span it starts in (so a span reads fewer than 2S
// edges), and a heavier row is cut at every multiple of S.  Its row-end bits
// (one 32-bit word per 32 edges) say where rows close, its window ranks and
// list of non-empty rows turn a close into a row id, so the edge loop reads
// no row pointers and searches for no row, and a row's degree is the distance
// between two closes.  A span stores the pieces of heavy rows that it holds
// with plain stores -- at most two: the end of one that started earlier
// (slot 2w) and the start of one that runs on (slot 2w+1) -- so nothing on
// the edge path waits on another warp or on an atomic unit, and
// k_agg_span_fix sums every heavy row's pieces in edge order once this grid
// has finished.  Max, whose merge is exact in any order, instead folds all of
// a row's pieces into the tail slot of its first span with 64-bit max
// reductions.  Warps past the last span write the empty rows.
#ifndef GNN_SPAN_U
#define GNN_SPAN_U 4
#endif
// minimum resident warps per SM / 8, and threads per block
#ifndef GNN_SPAN_MINB
#define GNN_SPAN_MINB 4
#endif
// the same for max / min on fp32 rows: 64 registers (32 warps per SM) with
// a 16-byte spill measured faster than 80 registers at 24 warps (R-MAT scale
// 17 max 0.178 -> 0.173 ms, min 0.176 -> 0.172)
#ifndef GNN_SPAN_EXT_MINB
#define GNN_SPAN_EXT_MINB 4
#endif
#ifndef GNN_SPAN_BLOCK
#define GNN_SPAN_BLOCK 64
#endif
constexpr int kSpanBlock = GNN_SPAN_BLOCK;
constexpr int32_t kEmptyRowsPerWarp = 256;

// arr[i] for a run-time i without local memory (a chain of selects)
template <int N, class V>
__device__ __forceinline__ V pick(const V (&arr)[N], int i) {
    V r = arr[0];
#pragma unroll
    for (int k = 1; k < N; ++k)
        if (i == k) r = arr[k];
    return r;
}

// Row-end bits of edges [e, e+32) (bit i for edge e+i), e not necessarily
// a multiple of 32.
__device__ __forceinline__ uint32_t end_bits(const uint32_t *__restrict__ flags, int32_t n_win,
                                             int32_t e) {
    const int32_t lo = e >> 5, sh = e & 31;
    const uint32_t w0 = __ldg(flags + lo);
    if (sh == 0) return w0;
    const uint32_t w1 = lo + 1 < n_win ? __ldg(flags + lo + 1) : 0u;
    return __funnelshift_r(w0, w1, sh);
}

// Zero rows (argmax -1) for the empty rows among [q*256, (q+1)*256).
template <int OP>
__device__ __forceinline__ void write_empty_rows(const AggArgs &a, int32_t q, int lane) {
    const unsigned FULL = 0xffffffffu;
    constexpr int NB = kEmptyRowsPerWarp / 32;
    const int32_t r0 = q * kEmptyRowsPerWarp;
    bool empty[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int32_t r = r0 + 32 * i + lane;
        empty[i] = r < a.n_rows && __ldg(a.rowptr + r + 1) == __ldg(a.rowptr + r);
    }
    const int32_t n4 = a.F / 4;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        unsigned m = __ballot_sync(FULL, empty[i]);
        while (m) {
            const int32_t r = r0 + 32 * i + __ffs(m) - 1;
            m &= m - 1;
            float4 *y = reinterpret_cast<float4 *>(a.Y + (size_t)r * a.F);
            for (int32_t c = lane; c < n4; c += 32) y[c] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (is_ext(OP) && a.argmax) {
                int4 *am = reinterpret_cast<int4 *>(a.argmax + (size_t)r * a.F);
                for (int32_t c = lane; c < n4; c += 32) am[c] = make_int4(-1, -1, -1, -1);
            }
        }
    }
}

// Piece (or chunk) records of the edge-span path: per lane NV fp32 partial
// sums, or for max NV 64-bit words (key << 32) | ~source_id, whose unsigned
// maximum is the packed (value, index) merge of IO-aware GNN layers,
// Appendix D.1 (ties to the smaller id).
template <int OP, class T>
__device__ __forceinline__ void store_piece(const AggArgs &a, float *base, int64_t slot,
                                            const Acc<OP, T, 1> &acc, int lane) {
    constexpr int NV = Chunk<T>::N;
    const int64_t off = slot * a.F + (int64_t)lane * NV;
    if (is_ext(OP)) {
        ulonglong2 *dst = reinterpret_cast<ulonglong2 *>(reinterpret_cast<unsigned long long *>(base) + off);
#pragma unroll
        for (int k = 0; k < NV; k += 2) {
            ulonglong2 w;
            w.x = ((unsigned long long)acc.key(0, k) << 32) | (0xFFFFFFFFu - (uint32_t)acc.idx[0][k]);
            w.y = ((unsigned long long)acc.key(0, k + 1) << 32) | (0xFFFFFFFFu - (uint32_t)acc.idx[0][k + 1]);
            dst[k / 2] = w;
        }
    } else {
        float4 *dst = reinterpret_cast<float4 *>(base + off);
#pragma unroll
        for (int k = 0; k < NV; k += 4)
            dst[k / 4] = make_float4(acc.v[0][k], acc.v[0][k + 1], acc.v[0][k + 2], acc.v[0][k + 3]);
    }
}

// Max: every piece of a heavy row is folded into one slot with 64-bit
// reductions (the merge is exact and order-free); the warp does not wait.
template <int OP, class T>
__device__ __forceinline__ void fold_max_piece(const AggArgs &a, int64_t slot,
                                               const Acc<OP, T, 1> &acc, int lane) {
    constexpr int NV = Chunk<T>::N;
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(a.carry) + slot * a.F + (int64_t)lane * NV;
#pragma unroll
    for (int k = 0; k < NV; ++k)
        atomicMax(dst + k, ((unsigned long long)acc.key(0, k) << 32) | (0xFFFFFFFFu - (uint32_t)acc.idx[0][k]));
}

// One lane's share of a piece record, loaded ahead of merging.
template <int OP, class T>
struct PieceVal {
    static constexpr int NV = Chunk<T>::N;
    static constexpr int NW = is_ext(OP) ? NV / 2 : NV / 4;  // 16-byte words
    uint4 w[NW];
    __device__ __forceinline__ void load(const AggArgs &a, const float *base, int64_t slot, int lane,
                                         bool bypass_l1) {
        const int64_t off = slot * a.F + (int64_t)lane * NV;
        const uint4 *src = is_ext(OP)
                               ? reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned long long *>(base) + off)
                               : reinterpret_cast<const uint4 *>(base + off);
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = bypass_l1 ? ldcg16(src + i) : ldg16(src + i);
    }
    // clear the record just read (the workspace is left zero-filled)
    __device__ __forceinline__ static void clear(const AggArgs &a, float *base, int64_t slot, int lane) {
        const int64_t off = slot * a.F + (int64_t)lane * NV;
        uint4 *dst = is_ext(OP)
                         ? reinterpret_cast<uint4 *>(reinterpret_cast<unsigned long long *>(base) + off)
                         : reinterpret_cast<uint4 *>(base + off);
#pragma unroll
        for (int i = 0; i < NW; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    // acc := acc (+) this, in that order
    __device__ __forceinline__ void merge_into(Acc<OP, T, 1> &acc) const {
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            if (is_ext(OP)) {
                const unsigned long long p0 = ((unsigned long long)w[i].y << 32) | w[i].x;
                const unsigned long long p1 = ((unsigned long long)w[i].w << 32) | w[i].z;
#pragma unroll
                for (int z = 0; z < 2; ++z) {
                    const int k = 2 * i + z;
                    const unsigned long long p = z ? p1 : p0;
                    const unsigned long long cur =
                        ((unsigned long long)acc.key(0, k) << 32) | (0xFFFFFFFFu - (uint32_t)acc.idx[0][k]);
                    if (p > cur) acc.set_packed(0, k, p);
                }
            } else {
                acc.v[0][4 * i] += __uint_as_float(w[i].x);
                acc.v[0][4 * i + 1] += __uint_as_float(w[i].y);
                acc.v[0][4 * i + 2] += __uint_as_float(w[i].z);
                acc.v[0][4 * i + 3] += __uint_as_float(w[i].w);
            }
        }
    }
};

// WT = false: unit edge weights and row factor 1 (segment sum / mean / max);
// WT = true: the SpMM's per-edge weights and row factors.
template <int OP, class T, bool WT>
__device__ __forceinline__ void agg_span_one(const AggArgs &a, const int32_t w, const int lane) {
    constexpr int U = GNN_SPAN_U;
    const unsigned FULL = 0xffffffffu;
    if (w >= a.n_spans) {
        if (w - a.n_spans < (a.n_rows + kEmptyRowsPerWarp - 1) / kEmptyRowsPerWarp)
            write_empty_rows<OP>(a, w - a.n_spans, lane);
        return;
    }
    const int32_t b0 = __ldg(a.sp_begin + w), b1 = __ldg(a.sp_begin + w + 1);
    if (b0 >= b1) return;
    const int32_t n_win = (int32_t)((a.nnz + 31) >> 5);
    const bool weighted = WT && (a.values || a.col_mode != COL_ONE);
    const bool rsq = WT && a.row_mode == ROW_RSQRT;

    // first window's column ids (the next window's are fetched one ahead)
    int32_t c_cur = b0 + lane < b1 ? ld_col(a.colidx + b0 + lane) : 0;
    int32_t c_nxt = b0 + 32 + lane < b1 ? ld_col(a.colidx + b0 + 32 + lane) : 0;
    // rank of the row holding b0 = row ends before b0
    const uint32_t wb0 = __ldg(a.win_flags + (b0 >> 5));
    const int32_t k0 = __ldg(a.win_rowbase + (b0 >> 5)) + __popc(wb0 & ((1u << (b0 & 31)) - 1u));
    // a span that starts inside a row starts inside a heavy row; that row's
    // piece here goes to slot 2w, a heavy row that starts here and runs on
    // leaves its first piece in slot 2w+1 (max: every piece of a row goes to
    // the tail slot of the span the row starts in)
    bool head = b0 > 0 && !((__ldg(a.win_flags + ((b0 - 1) >> 5)) >> ((b0 - 1) & 31)) & 1u);
    const int64_t max_head_slot =
        (is_ext(OP) && head) ? 2 * (int64_t)(__ldg(a.win_rowstart + (b0 >> 5)) >> a.span_shift) + 1 : 0;
    // lane l holds the id (and row factor) of the row of rank k0 + kofs + l
    int32_t kofs = 0;
    int32_t rid = k0 + lane < a.n_rows ? __ldg(a.ne_rows + k0 + lane) : 0;
    float w_cur = (weighted && b0 + lane < b1) ? edge_weight(a, b0 + lane, c_cur) : 1.f;
    float rf = rsq ? __ldg(a.dinv_in + rid) : 1.f;

    Acc<OP, T, 1> acc;
    acc.reset();
    int32_t k = 0;     // rows closed so far in this span
    int32_t rs = b0;   // first edge of the open row
    uint32_t last_closed = 1u;
#pragma unroll 1
    for (int32_t cb = b0; cb < b1; cb += 32) {
        const int n = min(32, b1 - cb);
        const uint32_t bits_all = end_bits(a.win_flags, n_win, cb);
        last_closed = (bits_all >> (n - 1)) & 1u;
        const uint32_t bits = n == 32 ? bits_all : bits_all & ((1u << n) - 1u);
#pragma unroll 1
        for (int u0 = 0; u0 < n; u0 += U) {
            uint4 xv[U];
            int32_t jv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                jv[u] = __shfl_sync(FULL, c_cur, (u0 + u) & 31);
                if (u0 + u < n) xv[u] = ldg16(a.X + (size_t)jv[u] * 32 + lane);
            }
            const uint32_t gb = (bits >> u0) & ((1u << U) - 1u);
            if (gb == 0 && u0 + U <= n) {
                // no row closes inside this group
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                    acc.add(&xv[u], ww, jv[u]);
                }
                continue;
            }
            if (!head) {
                // rows close here, all of them whole rows of this span: keep
                // the ids of the next U ranks in the lane window
                if (k - kofs > 32 - U) {
                    kofs = k;
                    rid = k0 + kofs + lane < a.n_rows ? __ldg(a.ne_rows + k0 + kofs + lane) : 0;
                    if (rsq) rf = __ldg(a.dinv_in + rid);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (u0 + u < n) {
                        const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                        acc.add(&xv[u], ww, jv[u]);
                        if ((gb >> u) & 1u) {
                            const int32_t e = cb + u0 + u;
                            const int32_t r = __shfl_sync(FULL, rid, k - kofs);
                            const float f = rsq ? __shfl_sync(FULL, rf, k - kofs) : 1.f;
                            store_row_f<OP, T, 1>(a, r, e - rs + 1, f, acc, lane);
                            acc.reset();
                            ++k;
                            rs = e + 1;
                        }
                    }
                }
                continue;
            }
            // the group where the heavy row this span started inside closes
#pragma unroll 1
            for (int u = 0; u < U && u0 + u < n; ++u) {
                const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                const uint4 x = pick(xv, u);
                acc.add(&x, ww, pick(jv, u));
                if ((gb >> u) & 1u) {
                    const int32_t e = cb + u0 + u;
                    if (head) {
                        if constexpr (is_ext(OP)) {
                            fold_max_piece<OP, T>(a, max_head_slot, acc, lane);
                        } else {
                            store_piece<OP, T>(a, a.carry, 2 * (int64_t)w, acc, lane);
                        }
                        head = false;
                    } else {
                        if (k - kofs == 32) {
                            kofs += 32;
                            rid = k0 + kofs + lane < a.n_rows ? __ldg(a.ne_rows + k0 + kofs + lane) : 0;
                            if (rsq) rf = __ldg(a.dinv_in + rid);
                        }
                        const int32_t r = __shfl_sync(FULL, rid, k - kofs);
                        const float f = rsq ? __shfl_sync(FULL, rf, k - kofs) : 1.f;
                        store_row_f<OP, T, 1>(a, r, e - rs + 1, f, acc, lane);
                    }
                    acc.reset();
                    ++k;
                    rs = e + 1;
                }
            }
        }
        // advance the column window
        c_cur = c_nxt;
        const int32_t en = cb + 64 + lane;
        c_nxt = en < b1 ? ld_col(a.colidx + en) : 0;
        if (weighted) w_cur = cb + 32 + lane < b1 ? edge_weight(a, cb + 32 + lane, c_cur) : 1.f;
    }
    // a heavy row reaches past this span: leave its piece
    if (!last_closed) {
        if constexpr (is_ext(OP)) {
            fold_max_piece<OP, T>(a, head ? max_head_slot : 2 * (int64_t)w + 1, acc, lane);
        } else {
            store_piece<OP, T>(a, a.carry, 2 * (int64_t)w + (head ? 0 : 1), acc, lane);
        }
    }
}

// Work items of the span kernels: the spans, then the empty-row blocks.
__device__ __forceinline__ int32_t span_items(const AggArgs &a) {
    return a.n_spans + (a.n_rows + kEmptyRowsPerWarp - 1) / kEmptyRowsPerWarp;
}

// One warp per span (the grid covers every span).  The body is a device
// function called from a loop: measured on GB300 with fp32 rows at R-MAT
// scale 17, this form of the same code runs segment sum in 0.113 ms against
// 0.121 for the body written inline in the kernel (one resident wave of
// warps striding over the spans was no faster).
template <int OP, class T, bool WT>
__global__ void __launch_bounds__(kSpanBlock, ((!is_ext(OP) && sizeof(T) == 4) ? GNN_SPAN_MINB : (is_ext(OP) && sizeof(T) == 4) ? GNN_SPAN_EXT_MINB : GNN_SPAN_MINB - 1) * 256 / kSpanBlock)
k_agg_span(AggArgs a) {
    // let the finalising kernel start its launch while this grid drains
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int32_t nw = (int32_t)(((int64_t)gridDim.x * blockDim.x) >> 5);
    const int32_t items = span_items(a);
    for (int32_t w = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5); w < items; w += nw)
        agg_span_one<OP, T, WT>(a, w, lane);
}

// Lean variant of k_agg_span for the sum-like ops (SpMM, sum, mean): the
// same spans, row-end bits, row ranks and piece slots, but one loop over
// groups of U edges with the row closes tested edge by edge, instead of
// separate close-free, whole-row and head-piece paths.  Fewer values stay
// live across the loop, so more warps fit on an SM; the kernel is bound by
// the feature rows in flight per SM (warps x U).
// rows in flight per lane, and resident 64-thread blocks per SM asked of the
// compiler (U = 8 at 12 blocks fits 80 registers without spills: 24 warps x
// 8 rows in flight per SM, against 28 x 4 for k_agg_span)
#ifndef GNN_LEAN_U
#define GNN_LEAN_U 4
#endif
#ifndef GNN_LEAN_MINB
#define GNN_LEAN_MINB 16
#endif
#ifndef GNN_SPAN_LEAN
#define GNN_SPAN_LEAN 1
#endif

template <int OP, class T, bool WT>
__global__ void __launch_bounds__(kSpanBlock, GNN_LEAN_MINB * 64 / kSpanBlock) k_agg_span_lean(AggArgs a) {
    static_assert(!is_ext(OP), "sum-like ops only");
    constexpr int U = GNN_LEAN_U;
    static_assert(32 % U == 0, "groups tile a 32-edge window");
    const unsigned FULL = 0xffffffffu;
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int32_t w = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (w >= a.n_spans) {
        if (w - a.n_spans < (a.n_rows + kEmptyRowsPerWarp - 1) / kEmptyRowsPerWarp)
            write_empty_rows<OP>(a, w - a.n_spans, lane);
        return;
    }
    const int32_t b0 = __ldg(a.sp_begin + w), b1 = __ldg(a.sp_begin + w + 1);
    if (b0 >= b1) return;
    const int32_t n_win = (int32_t)((a.nnz + 31) >> 5);
    const bool weighted = WT && (a.values || a.col_mode != COL_ONE);
    const bool rsq = WT && a.row_mode == ROW_RSQRT;

    int32_t c_cur = b0 + lane < b1 ? ld_col(a.colidx + b0 + lane) : 0;
    int32_t c_nxt = b0 + 32 + lane < b1 ? ld_col(a.colidx + b0 + 32 + lane) : 0;
    // rank of the row holding b0; a span that starts inside a row starts
    // inside a heavy row, whose piece here goes to slot 2w
    const uint32_t wb0 = __ldg(a.win_flags + (b0 >> 5));
    const int32_t k0 = __ldg(a.win_rowbase + (b0 >> 5)) + __popc(wb0 & ((1u << (b0 & 31)) - 1u));
    bool head = b0 > 0 && !((__ldg(a.win_flags + ((b0 - 1) >> 5)) >> ((b0 - 1) & 31)) & 1u);
    int32_t kofs = 0;  // lane l holds the id (and row factor) of the row of rank k0 + kofs + l
    int32_t rid = k0 + lane < a.n_rows ? __ldg(a.ne_rows + k0 + lane) : 0;
    float w_cur = (weighted && b0 + lane < b1) ? edge_weight(a, b0 + lane, c_cur) : 1.f;
    float rf = rsq ? __ldg(a.dinv_in + rid) : 1.f;
    const uint4 *__restrict__ Xl = a.X + lane;

    Acc<OP, T, 1> acc;
    acc.reset();
    int32_t k = 0;    // rows closed so far in this span
    int32_t rs = b0;  // first edge of the open row
    uint32_t last_closed = 1u;
#pragma unroll 1
    for (int32_t cb = b0; cb < b1; cb += 32) {
        const int n = min(32, b1 - cb);
        const uint32_t bits_all = end_bits(a.win_flags, n_win, cb);
        last_closed = (bits_all >> (n - 1)) & 1u;
#pragma unroll 1
        for (int u0 = 0; u0 < n; u0 += U) {
            uint4 xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t j = __shfl_sync(FULL, c_cur, (u0 + u) & 31);
                if (u0 + u < n) xv[u] = ldg16(Xl + (size_t)j * 32);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u0 + u >= n) break;
                const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                acc.add(&xv[u], ww, 0);
                if ((bits_all >> (u0 + u)) & 1u) {
                    const int32_t e = cb + u0 + u;
                    if (head) {
                        store_piece<OP, T>(a, a.carry, 2 * (int64_t)w, acc, lane);
                        head = false;
                    } else {
                        if (k - kofs == 32) {
                            kofs += 32;
                            rid = k0 + kofs + lane < a.n_rows ? __ldg(a.ne_rows + k0 + kofs + lane) : 0;
                            if (rsq) rf = __ldg(a.dinv_in + rid);
                        }
                        const int32_t r = __shfl_sync(FULL, rid, k - kofs);
                        const float f = rsq ? __shfl_sync(FULL, rf, k - kofs) : 1.f;
                        store_row_f<OP, T, 1>(a, r, e - rs + 1, f, acc, lane);
                    }
                    acc.reset();
                    ++k;
                    rs = e + 1;
                }
            }
        }
        // advance the column window
        c_cur = c_nxt;
        const int32_t en = cb + 64 + lane;
        c_nxt = en < b1 ? ld_col(a.colidx + en) : 0;
        if (weighted) w_cur = cb + 32 + lane < b1 ? edge_weight(a, cb + 32 + lane, c_cur) : 1.f;
    }
    // a heavy row reaches past this span: leave its piece
    if (!last_closed) store_piece<OP, T>(a, a.carry, 2 * (int64_t)w + (head ? 0 : 1), acc, lane);
}

// Ring variant of the span kernels: the same spans, row-end bits, row ranks
// and piece slots as k_agg_span, but the feature rows travel global ->
// shared memory by 16-byte cp.async copies into a per-warp ring of P groups
// of GNN_RING_G edges, instead of into registers.  Lane l copies bytes
// [16l, 16l+16) of every row and later reads back exactly those bytes, so its
// own cp.async.wait_group orders the data (no barrier, no mbarrier).  Rows in
// flight hold no registers: a warp keeps between (P-1)*G and P*G rows in
// flight at all times, where the register-gather kernels drain their U rows
// before each group is summed.  Measured on GB300 (G = 4): R-MAT scale 22
// SpMM with bf16 rows 4.89 -> 3.81 ms at P = 3 (3.87 at P = 2, 3.88 at
// P = 4 with 24 warps per SM, 3.96 for G = 2, P = 6); R-MAT scale 17 segment
// sum with fp32 rows 0.115 -> 0.091 ms at P = 2 (0.093 at P = 3).
#ifndef GNN_RING_G
#define GNN_RING_G 4
#endif
#ifndef GNN_RING_P_BF16
#define GNN_RING_P_BF16 3
#endif
#ifndef GNN_RING_P_F32
#define GNN_RING_P_F32 2
#endif
#ifndef GNN_RING_MINB
#define GNN_RING_MINB 16
#endif
#ifndef GNN_RING_EXT_MINB
#define GNN_RING_EXT_MINB 16
#endif
// 0: off (register-gather span kernels); 1: on
#ifndef GNN_SPAN_RING
#define GNN_SPAN_RING 1
#endif
// groups of G edges without a row end summed on a path without per-edge tests
#ifndef GNN_RING_FAST
#define GNN_RING_FAST 1
#endif
// max / min on the ring kernel (1) or on k_agg_span (0)
#ifndef GNN_RING_EXT
#define GNN_RING_EXT 1
#endif
template <class T>
__host__ __device__ constexpr int ring_groups() { return sizeof(T) == 2 ? GNN_RING_P_BF16 : GNN_RING_P_F32; }
template <class T>
__host__ __device__ constexpr int ring_bytes_per_warp() { return GNN_RING_G * ring_groups<T>() * 512; }

// 16-byte copy global -> shared around L1 (.cg): copying through L1 (.ca)
// measured slower on GB300 (R-MAT scale 22 SpMM 5.99 against 3.81 ms,
// scale 17 sum 0.122 against 0.093 ms), and so did an L2 priority by source
// out-degree through .L2::cache_hint (evict_first below d_out 16 or 48,
// evict_last from 48, 64 or 128: 4.68-4.96 ms against 3.81)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

template <int OP, class T, bool WT>
__global__ void __launch_bounds__(kSpanBlock, (is_ext(OP) ? GNN_RING_EXT_MINB : GNN_RING_MINB) * 64 / kSpanBlock)
k_agg_span_ring(AggArgs a) {
    constexpr int G = GNN_RING_G, P = ring_groups<T>();
    static_assert(32 % G == 0 && 16 % G == 0 && P >= 2 && (P - 1) * G <= 32,
                  "groups tile a window; issue runs at most one window ahead");
    extern __shared__ __align__(16) uint4 ring_buf[];
    const unsigned FULL = 0xffffffffu;
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const int32_t w = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (w >= a.n_spans) {
        if (w - a.n_spans < (a.n_rows + kEmptyRowsPerWarp - 1) / kEmptyRowsPerWarp)
            write_empty_rows<OP>(a, w - a.n_spans, lane);
        return;
    }
    const int32_t b0 = __ldg(a.sp_begin + w), b1 = __ldg(a.sp_begin + w + 1);
    if (b0 >= b1) return;
    const int32_t len = b1 - b0;
    const int32_t n_win = (int32_t)((a.nnz + 31) >> 5);
    const bool weighted = WT && (a.values || a.col_mode != COL_ONE);
    const bool rsq = WT && a.row_mode == ROW_RSQRT;
    // this lane's 16 bytes of ring slot s: ring0 + 512 * s
    const uint32_t ring0 = su32(ring_buf + (threadIdx.x >> 5) * (ring_bytes_per_warp<T>() / 16) + lane);
    const uint4 *__restrict__ Xl = a.X + lane;

    // column ids of the window being summed (c_cur) and of the next (c_nxt)
    int32_t c_cur = lane < len ? ld_col(a.colidx + b0 + lane) : 0;
    int32_t c_nxt = 32 + lane < len ? ld_col(a.colidx + b0 + 32 + lane) : 0;
    // copy the rows of group q (edges b0 + qG ..) into slot group qs; cw is
    // the span offset of c_cur's window (the group lies in it or the next)
    auto issue = [&](int32_t q, int qs, int32_t cw) {
        const int32_t t0 = q * G;
        const int32_t cols = t0 >= cw + 32 ? c_nxt : c_cur;
#pragma unroll
        for (int u = 0; u < G; ++u) {
            const int32_t j = __shfl_sync(FULL, cols, (t0 + u) & 31);
            if (t0 + u < len) cp_async16(ring0 + (uint32_t)(qs * G + u) * 512u, Xl + (size_t)j * 32);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int q = 0; q < P - 1; ++q) issue(q, q, 0);

    const uint32_t wb0 = __ldg(a.win_flags + (b0 >> 5));
    const int32_t k0 = __ldg(a.win_rowbase + (b0 >> 5)) + __popc(wb0 & ((1u << (b0 & 31)) - 1u));
    // a span that starts inside a row starts inside a heavy row; that row's
    // piece here goes to slot 2w (max: every piece of a row is folded into
    // the tail slot of the span the row starts in)
    bool head = b0 > 0 && !((__ldg(a.win_flags + ((b0 - 1) >> 5)) >> ((b0 - 1) & 31)) & 1u);
    const int64_t max_head_slot =
        (is_ext(OP) && head) ? 2 * (int64_t)(__ldg(a.win_rowstart + (b0 >> 5)) >> a.span_shift) + 1 : 0;
    int32_t kofs = 0;  // lane l holds the id (and row factor) of the row of rank k0 + kofs + l
    int32_t rid = k0 + lane < a.n_rows ? __ldg(a.ne_rows + k0 + lane) : 0;
    float w_cur = (weighted && lane < len) ? edge_weight(a, b0 + lane, c_cur) : 1.f;
    float w_nxt = 1.f;
    float rf = rsq ? __ldg(a.dinv_in + rid) : 1.f;

    Acc<OP, T, 1> acc;
    acc.reset();
    int32_t k = 0;    // rows closed so far in this span
    int32_t rs = b0;  // first edge of the open row
    uint32_t last_closed = 1u;
    int32_t q = 0;    // group summed next
    int qs_c = 0, qs_i = P - 1;
#pragma unroll 1
    for (int32_t cw = 0; cw < len; cw += 32) {
        const int32_t cb = b0 + cw;
        const int n = min(32, len - cw);
        const uint32_t bits_all = end_bits(a.win_flags, n_win, cb);
        last_closed = (bits_all >> (n - 1)) & 1u;
#pragma unroll 1
        for (int u0 = 0; u0 < n; u0 += G, ++q) {
            issue(q + P - 1, qs_i, cw);
            qs_i = qs_i + 1 == P ? 0 : qs_i + 1;
            // the next window's weights, once its column ids have arrived
            if (weighted && u0 == 16)
                w_nxt = cw + 32 + lane < len ? edge_weight(a, cb + 32 + lane, c_nxt) : 1.f;
            cp_async_wait<P - 1>();
            uint4 xv[G];
#pragma unroll
            for (int u = 0; u < G; ++u) xv[u] = lds16(ring0 + (uint32_t)(qs_c * G + u) * 512u);
            qs_c = qs_c + 1 == P ? 0 : qs_c + 1;
            if (GNN_RING_FAST && u0 + G <= n && ((bits_all >> u0) & ((1u << G) - 1u)) == 0u) {
                // no row ends among these G edges: sum them without the tests
#pragma unroll
                for (int u = 0; u < G; ++u) {
                    const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                    const int32_t j = is_ext(OP) ? __shfl_sync(FULL, c_cur, (u0 + u) & 31) : 0;
                    acc.add(&xv[u], ww, j);
                }
                continue;
            }
#pragma unroll
            for (int u = 0; u < G; ++u) {
                if (u0 + u >= n) break;
                const float ww = weighted ? __shfl_sync(FULL, w_cur, (u0 + u) & 31) : 1.f;
                const int32_t j = is_ext(OP) ? __shfl_sync(FULL, c_cur, (u0 + u) & 31) : 0;
                acc.add(&xv[u], ww, j);
                if ((bits_all >> (u0 + u)) & 1u) {
                    const int32_t e = cb + u0 + u;
                    if (head) {
                        if constexpr (is_ext(OP)) fold_max_piece<OP, T>(a, max_head_slot, acc, lane);
                        else store_piece<OP, T>(a, a.carry, 2 * (int64_t)w, acc, lane);
                        head = false;
                    } else {
                        if (k - kofs == 32) {
                            kofs += 32;
                            rid = k0 + kofs + lane < a.n_rows ? __ldg(a.ne_rows + k0 + kofs + lane) : 0;
                            if (rsq) rf = __ldg(a.dinv_in + rid);
                        }
                        const int32_t r = __shfl_sync(FULL, rid, k - kofs);
                        const float f = rsq ? __shfl_sync(FULL, rf, k - kofs) : 1.f;
                        store_row_f<OP, T, 1>(a, r, e - rs + 1, f, acc, lane);
                    }
                    acc.reset();
                    ++k;
                    rs = e + 1;
                }
            }
        }
        // advance the column window (a window of fewer than 17 edges never
        // reached u0 == 16: its successor is past the span's end anyway)
        c_cur = c_nxt;
        c_nxt = cw + 64 + lane < len ? ld_col(a.colidx + cb + 64 + lane) : 0;
        w_cur = w_nxt;
    }
    // no copy may still target this warp's ring when the warp exits
    cp_async_wait<0>();
    // a heavy row reaches past this span: leave its piece
    if (!last_closed) {
        if constexpr (is_ext(OP)) fold_max_piece<OP, T>(a, head ? max_head_slot : 2 * (int64_t)w + 1, acc, lane);
        else store_piece<OP, T>(a, a.carry, 2 * (int64_t)w + (head ? 0 : 1), acc, lane);
    }
}

// Finalise heavy rows (degree > S).  Such a row's edges lie in spans
// s0..s1 and it left one piece in each: the tail piece of span s0 (slot
// 2*s0+1), then the head pieces of spans s0+1..s1 (slots 2*s), in edge order
// (max: all folded into slot 2*s0+1, which is cleared again for the next
// call's reductions; the sum pieces are plain scratch, written before read).
// A persistent grid of warps strides over the prepared work items, each the
// pieces [16c, 16c+16) of one row, and sums them in edge order.  A row with
// one item is stored at once; otherwise each item leaves its chunk sum in the
// slot of its first piece, and the last of the row's items to finish (a
// ticket, no spinning) sums the chunk sums in order and stores the row -- so
// every sum is independent of scheduling.
__device__ __forceinline__ int64_t piece_slot(int32_t s0, int32_t p) {
    return p == 0 ? 2 * (int64_t)s0 + 1 : 2 * ((int64_t)s0 + p);
}

#ifndef GNN_FIX_BLOCKS
#define GNN_FIX_BLOCKS 4
#endif
constexpr int kFixBlocksPerSm = GNN_FIX_BLOCKS;
#ifndef GNN_FIX_WORDS
#define GNN_FIX_WORDS 4
#endif

template <int OP, class T>
__global__ void __launch_bounds__(256, kFixBlocksPerSm) k_agg_span_fix(AggArgs a) {
    // records in flight per lane: GNN_FIX_WORDS 16-byte words
    constexpr int PF = GNN_FIX_WORDS / PieceVal<OP, T>::NW > 0 ? GNN_FIX_WORDS / PieceVal<OP, T>::NW : 1;
    const unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int32_t nw = (int32_t)((gridDim.x * blockDim.x) >> 5);
    int32_t q = (int32_t)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    // the items are prep data: read them before waiting for the span kernel
    const int32_t n_items = __ldg(a.items_count);
    int4 it = q < n_items ? __ldg(a.items + q) : make_int4(0, 0, 0, 0);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (; q < n_items; q += nw) {
        const int32_t row = it.x, rb = it.y, re = it.z, cidx = it.w;
        if (q + nw < n_items) it = __ldg(a.items + q + nw);
        const int32_t s0 = rb >> a.span_shift;
        const int32_t np = ((re - 1) >> a.span_shift) - s0 + 1;
        const int32_t nch = (np + kFixChunk - 1) / kFixChunk;
        const int32_t p_lo = cidx * kFixChunk, p_hi = min(np, p_lo + kFixChunk);
        Acc<OP, T, 1> acc;
        acc.reset();
        if constexpr (is_ext(OP)) {
            // all pieces were folded into the first piece's slot
            if (cidx != 0) continue;
            PieceVal<OP, T> pv;
            pv.load(a, a.carry, piece_slot(s0, 0), lane, false);
            pv.merge_into(acc);
            PieceVal<OP, T>::clear(a, a.carry, piece_slot(s0, 0), lane);
            store_row<OP, T, 1>(a, row, re - rb, acc, lane);
            continue;
        }
        for (int32_t p0 = p_lo; p0 < p_hi; p0 += PF) {
            PieceVal<OP, T> pv[PF];
#pragma unroll
            for (int u = 0; u < PF; ++u) {
                const int32_t p = p0 + u;
                if (p < p_hi) pv[u].load(a, a.carry, piece_slot(s0, p), lane, false);
            }
#pragma unroll
            for (int u = 0; u < PF; ++u)
                if (p0 + u < p_hi) pv[u].merge_into(acc);
        }
        if (nch == 1) {
            store_row<OP, T, 1>(a, row, re - rb, acc, lane);
            continue;
        }
        // the chunk sum replaces the chunk's first piece (read above by this warp)
        const int32_t q0 = q - cidx;  // the row's first item: its ticket
        store_piece<OP, T>(a, a.carry, piece_slot(s0, p_lo), acc, lane);
        __threadfence();
        __syncwarp();
        int32_t t = 0;
        if (lane == 0) t = atomicAdd(a.tickets + q0, 1);
        t = __shfl_sync(FULL, t, 0);
        if (t != nch - 1) continue;
        __threadfence();
        acc.reset();
        for (int32_t c0 = 0; c0 < nch; c0 += PF) {
            PieceVal<OP, T> pv[PF];
#pragma unroll
            for (int u = 0; u < PF; ++u)
                if (c0 + u < nch) pv[u].load(a, a.carry, piece_slot(s0, (c0 + u) * kFixChunk), lane, true);
#pragma unroll
            for (int u = 0; u < PF; ++u)
                if (c0 + u < nch) pv[u].merge_into(acc);
        }
        store_row<OP, T, 1>(a, row, re - rb, acc, lane);
        if (lane == 0) a.tickets[q0] = 0;
    }
}

// FEAT mapping: one group of lpr lanes per destination row, lanes over
// feature chunks, neighbours in sequence (IO-aware GNN layers, Section 4.1,
// feature-parallel "dot-aggr" mapping).
template <class T, int CPL>
__global__ void __launch_bounds__(256) k_agg_feat(AggArgs a) {
    constexpr int U = CPL >= GNN_AGG_U ? 1 : GNN_AGG_U / CPL;
    const int lpr = a.lpr;
    const int lane = threadIdx.x & 31;
    const int gl = lane & (lpr - 1);
    const unsigned gmask = lpr == 32 ? 0xffffffffu : (((1u << lpr) - 1u) << (lane & ~(lpr - 1)));
    const int64_t r64 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / lpr;
    if (r64 >= a.n_rows) return;
    const int32_t r = (int32_t)r64;
    const int64_t b = __ldg(a.rowptr + r), e1 = __ldg(a.rowptr + r + 1);
    const bool weighted = a.values || a.col_mode != COL_ONE;
    Acc<AGG_WSUM, T, CPL> acc;
    acc.reset();
    for (int64_t cb = b; cb < e1; cb += lpr) {
        int32_t cj = (cb + gl < e1) ? __ldg(a.colidx + cb + gl) : 0;
        float cw = (weighted && cb + gl < e1) ? edge_weight(a, cb + gl, cj) : 1.f;
        int n = (int)((e1 - cb) < (int64_t)lpr ? (e1 - cb) : (int64_t)lpr);
        for (int u0 = 0; u0 < n; u0 += U) {
            uint4 xv[U][CPL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                int32_t j = __shfl_sync(gmask, cj, u0 + u, lpr);
                if (u0 + u < n) {
                    const uint4 *src = a.X + (int64_t)j * a.V + gl;
#pragma unroll
                    for (int c = 0; c < CPL; ++c) xv[u][c] = ldg16(src + c * lpr);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float wt = __shfl_sync(gmask, cw, u0 + u, lpr);
                if (u0 + u < n) acc.add(xv[u], wt, 0);
            }
        }
    }
    store_row<AGG_WSUM, T, CPL>(a, r, (int32_t)(e1 - b), acc, gl);
}

// NEIGH mapping: one warp per destination row, lanes over neighbours
// (gather); each lane reads UC consecutive 16-byte chunks of its neighbour,
// then a butterfly reduction across the warp per chunk (IO-aware GNN
// layers, Section 4.1, neighbour-parallel "dot-aggr" mapping).
template <class T>
__global__ void __launch_bounds__(256) k_agg_neigh(AggArgs a) {
    constexpr int NV = Chunk<T>::N;
    constexpr int UC = 4;
    const int lane = threadIdx.x & 31;
    const int64_t r64 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r64 >= a.n_rows) return;
    const int32_t r = (int32_t)r64;
    const int64_t b = __ldg(a.rowptr + r), e1 = __ldg(a.rowptr + r + 1);
    const bool weighted = a.values || a.col_mode != COL_ONE;
    const float s = row_factor(a, r, (int32_t)(e1 - b));
    for (int c0 = 0; c0 < a.V; c0 += UC) {
        float acc[UC][NV];
#pragma unroll
        for (int u = 0; u < UC; ++u)
#pragma unroll
            for (int k = 0; k < NV; ++k) acc[u][k] = 0.f;
        for (int64_t e = b + lane; e < e1; e += 32) {
            int32_t j = __ldg(a.colidx + e);
            float wt = weighted ? edge_weight(a, e, j) : 1.f;
            const uint4 *src = a.X + (int64_t)j * a.V + c0;
            uint4 xv[UC];
#pragma unroll
            for (int u = 0; u < UC; ++u)
                if (c0 + u < a.V) xv[u] = ldg16(src + u);
#pragma unroll
            for (int u = 0; u < UC; ++u) {
                if (c0 + u >= a.V) break;
                float f[NV];
                Chunk<T>::unpack(xv[u], f);
#pragma unroll
                for (int k = 0; k < NV; ++k) acc[u][k] = fmaf(wt, f[k], acc[u][k]);
            }
        }
#pragma unroll
        for (int u = 0; u < UC; ++u)
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                float v = acc[u][k];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[u][k] = v * s;
            }
        // lane u writes chunk c0+u
#pragma unroll
        for (int u = 0; u < UC; ++u) {
            if (lane == u && c0 + u < a.V) {
                float *dst = a.Y + (int64_t)r * a.F + (int64_t)(c0 + u) * NV;
#pragma unroll
                for (int k = 0; k < NV; k += 4)
                    *reinterpret_cast<float4 *>(dst + k) =
                        make_float4(acc[u][k], acc[u][k + 1], acc[u][k + 2], acc[u][k + 3]);
            }
        }
    }
}

// Backward of max / min (IO-aware GNN layers, Appendix D.1, the sparse
// scatter through the stored argmin): grad_X[arg[v,f], f] += grad_out[v,f].
// One thread per 4 consecutive (v, f) entries (F % 4 == 0): coalesced
// 16-byte reads of arg and grad_out, fp32 atomic adds the thread does not
// wait for.  An arg outside [-1, n_cols) sets the device error word and is
// skipped.
__global__ void k_ext_backward(const int4 *__restrict__ arg, const float4 *__restrict__ go, int64_t n4,
                               int32_t F, int32_t n_cols, float *__restrict__ gx, int32_t *err) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const int4 a = __ldg(arg + i);
        const float4 g = __ldg(go + i);
        const int32_t f = (int32_t)((i * 4) % F);
        const int32_t js[4] = {a.x, a.y, a.z, a.w};
        const float gs[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (js[k] < 0) continue;
            if (js[k] >= n_cols) { set_device_error(err, GNN_ERR_DEVICE_CHECK); continue; }
            atomicAdd(gx + (int64_t)js[k] * F + f + k, gs[k]);
        }
    }
}

// ------------------------------------------------------------- host side

struct AggShape {
    int32_t V, lpr, cpl, E;
};

static bool agg_shape(int32_t x_dtype, int32_t F, AggShape *s) {
    int nv = x_dtype == GNN_F32 ? 4 : 8;
    if (F <= 0 || F % nv) return false;
    int32_t V = F / nv;
    if (V < 8 || V > 256 || (V & (V - 1))) return false;
    s->V = V;
    s->lpr = V < 32 ? V : 32;
    s->cpl = V / s->lpr;
    s->E = kRunEdges;
    return true;
}

static int64_t n_workers_for(const gnn_csr *g, int32_t E) {
    int64_t n = (g->nnz + E - 1) / E;
    return n > 0 ? n : 1;
}

// Workspace, both AUTO schedules (a call uses one of them; the regions are
// disjoint so either may follow the other on the same workspace):
//   run tickets [n_runs] int32 and run slots [n_runs, F]     zero on entry and exit
//   item tickets [span_item_cap] int32                        zero on entry and exit
//   span piece slots [2 * n_spans, F]                         sums: written before read;
//                                                             max: zero on entry and exit
// Slots are fp32, or 64-bit (key, ~id) words for max.
struct AggWs {
    int32_t *run_tickets, *item_tickets;
    float *run_slots, *pieces;
    size_t bytes;
};

static AggWs agg_ws_layout(const gnn_csr *g, int32_t op, int32_t F, void *base) {
    const int64_t nr = n_workers_for(g, kRunEdges);
    const int64_t ns = std::max<int64_t>(n_spans_of(g->nnz), 1);
    const size_t wmul = (op == GNN_OP_MAX || op == GNN_OP_MIN) ? 2 : 1;
    Carver cv(base);
    AggWs L;
    L.run_tickets = cv.take<int32_t>((size_t)nr);
    L.item_tickets = cv.take<int32_t>((size_t)span_item_cap(g->nnz));
    L.run_slots = cv.take<float>((size_t)nr * F * wmul);
    L.pieces = cv.take<float>((size_t)2 * ns * F * wmul);
    L.bytes = cv.used;
    return L;
}

size_t agg_workspace_bytes(const gnn_csr *g, int32_t op, int32_t x_dtype_unused, int32_t F) {
    (void)x_dtype_unused;
    return agg_ws_layout(g, op, F, nullptr).bytes;
}

template <int OP, class T>
static void launch_auto(const AggArgs &a, int cpl, cudaStream_t s) {
    int64_t threads = a.n_workers * a.lpr;
    int blocks = (int)((threads + 255) / 256);
    if (a.lpr == 32) {
        switch (cpl) {
            case 1: k_agg_auto<OP, T, 1, 32><<<blocks, 256, 0, s>>>(a); break;
            case 2: k_agg_auto<OP, T, 2, 32><<<blocks, 256, 0, s>>>(a); break;
            case 4: k_agg_auto<OP, T, 4, 32><<<blocks, 256, 0, s>>>(a); break;
            default: k_agg_auto<OP, T, 8, 32><<<blocks, 256, 0, s>>>(a); break;
        }
    } else {
        k_agg_auto<OP, T, 1, 0><<<blocks, 256, 0, s>>>(a);
    }
}

template <class T>
static void launch_feat(const AggArgs &a, int cpl, cudaStream_t s) {
    int64_t threads = (int64_t)a.n_rows * a.lpr;
    int blocks = (int)((threads + 255) / 256);
    switch (cpl) {
        case 1: k_agg_feat<T, 1><<<blocks, 256, 0, s>>>(a); break;
        case 2: k_agg_feat<T, 2><<<blocks, 256, 0, s>>>(a); break;
        case 4: k_agg_feat<T, 4><<<blocks, 256, 0, s>>>(a); break;
        default: k_agg_feat<T, 8><<<blocks, 256, 0, s>>>(a); break;
    }
}

// The span kernel, then (if any span boundary exists) the kernel that
// finalises cut rows, launched as a programmatic dependent of the first so
// its launch overlaps the span kernel's last wave.
template <int OP, class T, bool WT>
static cudaError_t launch_span(const AggArgs &a, cudaStream_t s) {
    const int64_t warps =
        (int64_t)a.n_spans + ((int64_t)a.n_rows + kEmptyRowsPerWarp - 1) / kEmptyRowsPerWarp;
    const int span_blocks = (int)((warps * 32 + kSpanBlock - 1) / kSpanBlock);
    // bf16 rows: the lean kernel fits 32 warps per SM where k_agg_span's 72
    // registers fit 28 (R-MAT scale 22 SpMM 4.89 against 5.49 ms); fp32 rows
    // keep k_agg_span, which already fits 32 (scale 17: 0.136 against 0.146)
    const bool lean = GNN_SPAN_LEAN && !is_ext(OP) && sizeof(T) == 2;
    if (GNN_SPAN_RING && (GNN_RING_EXT || !is_ext(OP))) {
        // the rings of GNN_RING_MINB blocks must fit one SM's shared memory
        const cudaError_t attr = func_attr(reinterpret_cast<const void *>(k_agg_span_ring<OP, T, WT>),
                                           cudaFuncAttributePreferredSharedMemoryCarveout,
                                           cudaSharedmemCarveoutMaxShared);
        if (attr != cudaSuccess) return attr;
        const size_t smem = (size_t)(kSpanBlock / 32) * ring_bytes_per_warp<T>();
        k_agg_span_ring<OP, T, WT><<<span_blocks, kSpanBlock, smem, s>>>(a);
    } else if (lean) {
        k_agg_span_lean<(is_ext(OP) ? AGG_WSUM : OP), T, WT><<<span_blocks, kSpanBlock, 0, s>>>(a);
    } else {
        k_agg_span<OP, T, WT><<<span_blocks, kSpanBlock, 0, s>>>(a);
    }
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.n_spans <= 1) return e;
    // one resident wave of blocks strides over the work items
    const int64_t fix_blocks = std::min<int64_t>((span_item_cap(a.nnz) * 32 + 255) / 256,
                                                 (int64_t)sm_count() * kFixBlocksPerSm);
    if (fix_blocks <= 0) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)fix_blocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_agg_span_fix<OP, T>, a);
    note_launch();
    return e;
}

// Host checks shared by every aggregation entry point, in the order the
// header documents; nothing is launched before they pass.
gnn_status check_agg_args(const gnn_csr *g, const void *prep, int32_t norm, const void *X,
                          int32_t x_dtype, int32_t F, const float *Y, const int32_t *argmax,
                          int32_t mapping) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (!Y || (!X && g->n_cols > 0)) return GNN_ERR_INVALID_ARG;
    if (x_dtype != GNN_F32 && x_dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    if (norm < GNN_NORM_NONE || norm > GNN_NORM_BOTH) return GNN_ERR_INVALID_ARG;
    if (mapping < GNN_MAP_AUTO || mapping > GNN_MAP_NEIGH) return GNN_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Y) || (argmax && !aligned16(argmax))) return GNN_ERR_INVALID_ARG;
    AggShape sh;
    if (!agg_shape(x_dtype, F, &sh)) return GNN_ERR_UNSUPPORTED;
    if (norm != GNN_NORM_NONE && !prep) return GNN_ERR_INVALID_ARG;
    return GNN_OK;
}

gnn_status run_aggregate(const gnn_csr *g, const void *prep, int32_t op, int32_t norm,
                         const void *X, int32_t x_dtype, int32_t F, float *Y, int32_t *argmax,
                         int32_t mapping, void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_agg_args(g, prep, norm, X, x_dtype, F, Y, argmax, mapping);
    if (st != GNN_OK) return st;
    AggShape sh;
    agg_shape(x_dtype, F, &sh);
    if (g->n_rows == 0) return GNN_OK;

    AggArgs a{};
    a.rowptr = g->rowptr;
    a.colidx = g->colidx;
    a.values = (op == GNN_OP_SPMM) ? g->values : nullptr;
    a.X = static_cast<const uint4 *>(X);
    a.Y = Y;
    a.argmax = argmax;
    a.nnz = g->nnz;
    a.n_rows = g->n_rows;
    a.F = F;
    a.V = sh.V;
    a.lpr = sh.lpr;
    a.E = kRunEdges * GNN_AGG_RUNMUL;
    a.n_workers = n_workers_for(g, a.E);
    a.col_mode = COL_ONE;
    a.row_mode = ROW_ONE;
    if (prep) {
        prep_pointers(g, prep, &a.d_out, &a.dinv_in, &a.dinv_out);
        a.run_first_row = prep_run_table(g, prep);
    }
    if (op == GNN_OP_SPMM) {
        if (norm == GNN_NORM_LEFT) a.row_mode = ROW_RECIP;
        if (norm == GNN_NORM_RIGHT) a.col_mode = COL_RECIP;
        if (norm == GNN_NORM_BOTH) { a.row_mode = ROW_RSQRT; a.col_mode = COL_RSQRT; }
    }
    cudaStream_t s = as_stream(stream);
    const bool bf = x_dtype == GNN_BF16;

    if (op == GNN_OP_SPMM && mapping == GNN_MAP_FEAT) {
        if (bf) launch_feat<__nv_bfloat16>(a, sh.cpl, s); else launch_feat<float>(a, sh.cpl, s);
        note_launch();
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }
    if (op == GNN_OP_SPMM && mapping == GNN_MAP_NEIGH) {
        int blocks = (int)(((int64_t)g->n_rows * 32 + 255) / 256);
        if (bf) k_agg_neigh<__nv_bfloat16><<<blocks, 256, 0, s>>>(a);
        else k_agg_neigh<float><<<blocks, 256, 0, s>>>(a);
        note_launch();
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }

    size_t need = agg_workspace_bytes(g, op, x_dtype, F);
    if (!ws || ws_bytes < need) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    const AggWs L = agg_ws_layout(g, op, F, ws);
    a.carry = L.run_slots;
    a.tickets = L.run_tickets;

    if (prep && sh.V == 32) {
        prep_span_tables(g, prep, &a.win_flags, &a.win_rowbase, &a.ne_rows, &a.sp_begin, &a.items,
                         &a.items_count, &a.win_rowstart);
        a.E = span_edges(g->nnz);
        a.span_shift = span_shift(g->nnz);
        a.n_spans = (int32_t)n_spans_of(g->nnz);
        a.carry = L.pieces;
        a.tickets = L.item_tickets;
        const bool wt = a.values || a.col_mode != COL_ONE || a.row_mode != ROW_ONE;
        cudaError_t e;
        if (op == GNN_OP_MAX) e = bf ? launch_span<AGG_MAX, __nv_bfloat16, false>(a, s)
                                     : launch_span<AGG_MAX, float, false>(a, s);
        else if (op == GNN_OP_MIN) e = bf ? launch_span<AGG_MIN, __nv_bfloat16, false>(a, s)
                                          : launch_span<AGG_MIN, float, false>(a, s);
        else if (op == GNN_OP_MEAN) e = bf ? launch_span<AGG_MEAN, __nv_bfloat16, false>(a, s)
                                           : launch_span<AGG_MEAN, float, false>(a, s);
        else if (wt) e = bf ? launch_span<AGG_WSUM, __nv_bfloat16, true>(a, s)
                            : launch_span<AGG_WSUM, float, true>(a, s);
        else e = bf ? launch_span<AGG_WSUM, __nv_bfloat16, false>(a, s)
                    : launch_span<AGG_WSUM, float, false>(a, s);
        if (e != cudaSuccess) return cuda_status(e);
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }

    if (op == GNN_OP_MAX) {
        if (bf) launch_auto<AGG_MAX, __nv_bfloat16>(a, sh.cpl, s);
        else launch_auto<AGG_MAX, float>(a, sh.cpl, s);
    } else if (op == GNN_OP_MIN) {
        if (bf) launch_auto<AGG_MIN, __nv_bfloat16>(a, sh.cpl, s);
        else launch_auto<AGG_MIN, float>(a, sh.cpl, s);
    } else if (op == GNN_OP_MEAN) {
        if (bf) launch_auto<AGG_MEAN, __nv_bfloat16>(a, sh.cpl, s);
        else launch_auto<AGG_MEAN, float>(a, sh.cpl, s);
    } else {
        if (bf) launch_auto<AGG_WSUM, __nv_bfloat16>(a, sh.cpl, s);
        else launch_auto<AGG_WSUM, float>(a, sh.cpl, s);
    }
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

}  // namespace gnn

using namespace gnn;

extern "C" {

gnn_status gnn_spmm(const gnn_csr *g, const void *prep, int32_t norm, const void *X,
                    int32_t x_dtype, int32_t F, float *Y, int32_t mapping, void *ws,
                    size_t ws_bytes, void *stream) {
    return run_aggregate(g, prep, GNN_OP_SPMM, norm, X, x_dtype, F, Y, nullptr, mapping, ws,
                         ws_bytes, stream);
}

gnn_status gnn_segment_reduce_sum(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, void *ws,
                                  size_t ws_bytes, void *stream) {
    return run_aggregate(g, prep, GNN_OP_SUM, GNN_NORM_NONE, X, x_dtype, F, Y, nullptr,
                         GNN_MAP_AUTO, ws, ws_bytes, stream);
}

gnn_status gnn_segment_reduce_mean(const gnn_csr *g, const void *prep, const void *X,
                                   int32_t x_dtype, int32_t F, float *Y, void *ws,
                                   size_t ws_bytes, void *stream) {
    return run_aggregate(g, prep, GNN_OP_MEAN, GNN_NORM_NONE, X, x_dtype, F, Y, nullptr,
                         GNN_MAP_AUTO, ws, ws_bytes, stream);
}

gnn_status gnn_segment_reduce_max(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, int32_t *argmax,
                                  void *ws, size_t ws_bytes, void *stream) {
    return run_aggregate(g, prep, GNN_OP_MAX, GNN_NORM_NONE, X, x_dtype, F, Y, argmax,
                         GNN_MAP_AUTO, ws, ws_bytes, stream);
}

gnn_status gnn_segment_reduce_ext_backward(const int32_t *arg, int32_t n_rows, int32_t F,
                                           const float *grad_out, int32_t n_cols, float *grad_X,
                                           void *stream) {
    if (n_rows < 0 || n_cols < 0 || F <= 0 || F % 4) return F > 0 && F % 4 ? GNN_ERR_UNSUPPORTED : GNN_ERR_INVALID_ARG;
    const int64_t n = (int64_t)n_rows * F;
    if ((n > 0 && (!arg || !grad_out)) || (n_cols > 0 && !grad_X)) return GNN_ERR_INVALID_ARG;
    if (!aligned16(arg) || !aligned16(grad_out) || !aligned16(grad_X)) return GNN_ERR_INVALID_ARG;
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    if (n_cols > 0) {
        const cudaError_t e = cudaMemsetAsync(grad_X, 0, sizeof(float) * (size_t)n_cols * F, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (n == 0) return GNN_OK;
    const int64_t n4 = n / 4;
    const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)sm_count() * 16);
    k_ext_backward<<<blocks, 256, 0, s>>>(reinterpret_cast<const int4 *>(arg), reinterpret_cast<const float4 *>(grad_out),
                                          n4, F, n_cols, grad_X, err);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_segment_reduce_min(const gnn_csr *g, const void *prep, const void *X,
                                  int32_t x_dtype, int32_t F, float *Y, int32_t *argmin,
                                  void *ws, size_t ws_bytes, void *stream) {
    return run_aggregate(g, prep, GNN_OP_MIN, GNN_NORM_NONE, X, x_dtype, F, Y, argmin,
                         GNN_MAP_AUTO, ws, ws_bytes, stream);
}

}  // extern "C"
