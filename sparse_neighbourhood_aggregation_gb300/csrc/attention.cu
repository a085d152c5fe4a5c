// Steps a4 (fused GATv2 forward) and a5 (fused Graph Transformer attention,
// CSR path), plus the SIMT projection used for fp32 inputs.
//
// IO-aware GNN layers, Section 2.2 (iii) (GATv2 and GT scores), Section 3.2
// and Appendix D.2 (fused CSR forward: score, online softmax and weighted
// aggregate in one pass over the destination's adjacency list, logsumexp kept
// for the backward pass; no per-edge score, weight or message reaches HBM).
//
// GB300 design.  One warp is one worker.  The edge list is cut into runs of
// E edges (the prepared graph's run table, read at a stride); a warp owns the
// rows whose first edge lies in its run and processes each of them whole
// (light rows), so short rows of a power-law graph are packed many to a
// warp.  A row longer than E (heavy) is cut at run boundaries; every piece
// leaves its softmax state (running max, running sum, unnormalised
// accumulator) in a workspace slot, and the last piece to finish (ticket
// counter, no spinning) merges the pieces in edge order, so the result does
// not depend on scheduling.  A run can hold the last piece of one heavy row
// and the first piece of the next, so each run has two slots: 2w for a piece
// continued from an earlier run, 2w+1 for the first piece of a row it owns.
//
// Lane layout: lane l owns CPL consecutive 16-byte chunks of a feature row
// (8 bf16 or 4 fp32 channels per chunk); a head's channels sit on
// D / (CPL * chunk) adjacent lanes, whose partial scores are summed with
// xor-shuffles.  Scores are kept in base-2 units (scaled by log2 e) so each
// softmax weight is a single exp2.
//
// GATv2 score.  With LeakyReLU slope s, LReLU(x) = (1+s)/2 x + (1-s)/2 |x|,
// so  e_ij = A_l[i] + A_r[j] + sum_d a''_d |l_id + r_jd|  with
// A_l[i,h] = sum_d a'_hd l_id, A_r[j,h] = sum_d a'_hd r_jd, a' = (1+s)/2 a,
// a'' = (1-s)/2 a.  A_l and A_r are per-node scalars computed once after the
// projection; per edge and channel only an add and an |.| multiply-add
// remain (the plain definition would need add, multiply, max and
// multiply-add).
#include <algorithm>

#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);
const int32_t *prep_run_table(const gnn_csr *g, const void *prep);

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// attention run = kAttnRunMul runs of the prepared graph's run table
constexpr int kAttnRunMul = 4;
constexpr int kAttnE = kRunEdges * kAttnRunMul;
// edges whose rows are loaded before any of them is used (fewer when a lane
// holds more channels, to stay within registers)
template <int CPL>
struct AttnU {
    static constexpr int value = CPL == 1 ? 4 : (CPL == 2 ? 2 : 1);
};

enum AttnKind { ATT_GATV2 = 0, ATT_GT = 1 };

// floats per softmax-state slot: HD accumulator channels then (m, s) per
// head, rounded up to 16 bytes so every slot starts 16-byte aligned
__host__ __device__ __forceinline__ int64_t slot_stride(int32_t HD, int32_t heads) {
    return ((int64_t)HD + 2 * heads + 3) & ~(int64_t)3;
}

struct AttnArgs {
    const int32_t *rowptr;
    const int32_t *colidx;
    const int32_t *run_table;  // prepared graph's run table (E = kRunEdges) or null
    const uint4 *Sg;           // gathered score rows: GATv2 r = H W_r, GT K
    const uint4 *Vg;           // gathered value rows: GATv2 r, GT V
    const uint4 *Qd;           // destination rows: GATv2 l = H W_l, GT Q
    const float *Al;           // GATv2 [n, heads] base-2 linear part at the destination
    const float *Ar;           // GATv2 [n, heads] base-2 linear part at the source
    const float *coef;         // GATv2 [HD] (1-s)/2 a log2e; GT unused
    float qscale;              // GT: scale * log2e
    float *out;                // [n_rows, HD]
    float *lse;                // [n_rows, heads] or null
    float *slots;              // [2 n_workers, HD + 2 heads]
    int32_t *tickets;          // [n_workers], zero on entry and on exit
    int64_t nnz;
    int64_t n_workers;
    int32_t n_rows;
    int32_t HD, heads, D;
    int32_t nch;               // 16-byte chunks per feature row
};

template <class T>
struct Elt;
template <>
struct Elt<float> {
    static constexpr int N = 4;
};
template <>
struct Elt<__nv_bfloat16> {
    static constexpr int N = 8;
};

// Softmax state of one (row, head) as held by each lane of the head:
// running max m (base 2), running sum s of exp2(e - m), and the lane's
// channels of the unnormalised weighted sum.
template <int NC>
struct SmState {
    float m, s;
    float acc[NC];
    __device__ __forceinline__ void reset() {
        m = -INFINITY;
        s = 0.f;
#pragma unroll
        for (int k = 0; k < NC; ++k) acc[k] = 0.f;
    }
};

template <int KIND, class T, int CPL>
struct AttnLane {
    static constexpr int NV = Elt<T>::N;
    static constexpr int NC = CPL * NV;  // channels per lane
    int lane;
    bool active;    // owns channels
    int head;       // head of the lane's channels
    int lph;        // lanes per head
    float coef[KIND == ATT_GATV2 ? NC : 1];

    __device__ __forceinline__ float head_sum(float v) const {
        for (int o = lph >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    }
};

template <class T, int CPL>
__device__ __forceinline__ void load_row(const uint4 *base, int64_t row, int nch, int lane, bool active,
                                         uint4 *v) {
    const uint4 *p = base + row * nch + lane * CPL;
#pragma unroll
    for (int c = 0; c < CPL; ++c) v[c] = active ? ldg16(p + c) : make_uint4(0u, 0u, 0u, 0u);
}

template <class T, int CPL>
__device__ __forceinline__ void unpack_row(const uint4 *v, float *f) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) Chunk<T>::unpack(v[c], f + c * Elt<T>::N);
}

// Accumulate the edges [b, e) of destination row r into st.  dq: the
// destination's channels (l for GATv2, Q pre-scaled for GT); al: A_l[r,head].
template <int KIND, class T, int CPL>
__device__ __forceinline__ void attend_range(const AttnArgs &a, const AttnLane<KIND, T, CPL> &L,
                                             int32_t b, int32_t e, const float *dq, float al,
                                             SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    constexpr int U = AttnU<CPL>::value;
    const int lane = L.lane;
    for (int32_t wb = b; wb < e; wb += 32) {
        // column ids of the next (up to) 32 edges, one per lane
        const int32_t cj = (wb + lane < e) ? __ldg(a.colidx + wb + lane) : 0;
        const int nw = min(32, e - wb);
        for (int u0 = 0; u0 < nw; u0 += U) {
            uint4 sv[U][CPL];
            uint4 vv[KIND == ATT_GT ? U : 1][CPL];
            float ar[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int32_t j = __shfl_sync(0xffffffffu, cj, (u0 + u) & 31);
                const bool ok = u0 + u < nw;
                if (ok) {
                    load_row<T, CPL>(a.Sg, j, a.nch, lane, L.active, sv[u]);
                    if (KIND == ATT_GT) load_row<T, CPL>(a.Vg, j, a.nch, lane, L.active, vv[u]);
                    ar[u] = (KIND == ATT_GATV2 && L.active) ? __ldg(a.Ar + (int64_t)j * a.heads + L.head) : 0.f;
                }
            }
            float e2[U];
            float sf[U][KIND == ATT_GATV2 ? NC : 1];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float part = 0.f;
                if (KIND == ATT_GATV2) {
                    unpack_row<T, CPL>(sv[u], sf[u]);
#pragma unroll
                    for (int k = 0; k < NC; ++k) part = fmaf(L.coef[k], fabsf(dq[k] + sf[u][k]), part);
                } else {
                    float kf[NC];
                    unpack_row<T, CPL>(sv[u], kf);
#pragma unroll
                    for (int k = 0; k < NC; ++k) part = fmaf(dq[k], kf[k], part);
                }
                part = L.head_sum(part);
                e2[u] = (u0 + u < nw) ? (KIND == ATT_GATV2 ? part + al + ar[u] : part) : -INFINITY;
            }
            float mx = st.m;
#pragma unroll
            for (int u = 0; u < U; ++u) mx = fmaxf(mx, e2[u]);
            if (__any_sync(0xffffffffu, mx > st.m)) {
                const float sc = (mx > st.m) ? exp2f(st.m - mx) : 1.f;
                st.s *= sc;
#pragma unroll
                for (int k = 0; k < NC; ++k) st.acc[k] *= sc;
                st.m = mx;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (u0 + u < nw) {
                    const float p = exp2f(e2[u] - st.m);
                    st.s += p;
                    if (KIND == ATT_GATV2) {
#pragma unroll
                        for (int k = 0; k < NC; ++k) st.acc[k] = fmaf(p, sf[u][k], st.acc[k]);
                    } else {
                        float vf[NC];
                        unpack_row<T, CPL>(vv[u], vf);
#pragma unroll
                        for (int k = 0; k < NC; ++k) st.acc[k] = fmaf(p, vf[k], st.acc[k]);
                    }
                }
            }
        }
    }
}

template <int KIND, class T, int CPL>
__device__ __forceinline__ void store_final(const AttnArgs &a, const AttnLane<KIND, T, CPL> &L,
                                            int32_t r, const SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    if (!L.active) return;
    const float inv = st.s > 0.f ? 1.f / st.s : 0.f;
    float *o = a.out + (int64_t)r * a.HD + (int64_t)L.lane * NC;
#pragma unroll
    for (int k = 0; k < NC; k += 4)
        *reinterpret_cast<float4 *>(o + k) =
            make_float4(st.acc[k] * inv, st.acc[k + 1] * inv, st.acc[k + 2] * inv, st.acc[k + 3] * inv);
    if (a.lse && (L.lane % L.lph) == 0)
        a.lse[(int64_t)r * a.heads + L.head] = st.s > 0.f ? (st.m + log2f(st.s)) * kLn2 : -INFINITY;
}

// Load the destination-side data of row r: GATv2 l_r (unpacked) and A_l;
// GT Q_r pre-scaled by scale * log2 e.
template <int KIND, class T, int CPL>
__device__ __forceinline__ void load_dest(const AttnArgs &a, const AttnLane<KIND, T, CPL> &L,
                                          int32_t r, float *dq, float *al) {
    constexpr int NC = CPL * Elt<T>::N;
    uint4 v[CPL];
    load_row<T, CPL>(a.Qd, r, a.nch, L.lane, L.active, v);
    unpack_row<T, CPL>(v, dq);
    if (KIND == ATT_GT) {
#pragma unroll
        for (int k = 0; k < NC; ++k) dq[k] *= a.qscale;
        *al = 0.f;
    } else {
        *al = L.active ? __ldg(a.Al + (int64_t)r * a.heads + L.head) : 0.f;
    }
}

// A piece of heavy row r (edges of run w) leaves its state in slot 2w+1 (the
// row's first piece) or 2w (a later piece); the last piece to arrive merges
// the pieces of runs wa..wb in order and writes the row.
template <int KIND, class T, int CPL>
__device__ __forceinline__ void flush_piece(const AttnArgs &a, const AttnLane<KIND, T, CPL> &L,
                                            int64_t w, int32_t r, const SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    const int64_t stride = slot_stride(a.HD, a.heads);
    const int32_t rb = __ldg(a.rowptr + r), re = __ldg(a.rowptr + r + 1);
    const int64_t E = kAttnE;
    const int64_t wa = rb / E, wb = ((int64_t)re - 1) / E;
    float *slot = a.slots + (2 * w + (w == wa ? 1 : 0)) * stride;
    if (L.active) {
#pragma unroll
        for (int k = 0; k < NC; k += 4)
            __stcg(reinterpret_cast<float4 *>(slot + L.lane * NC + k),
                   make_float4(st.acc[k], st.acc[k + 1], st.acc[k + 2], st.acc[k + 3]));
        if ((L.lane % L.lph) == 0) {
            __stcg(slot + a.HD + 2 * L.head, st.m);
            __stcg(slot + a.HD + 2 * L.head + 1, st.s);
        }
    }
    __threadfence();
    __syncwarp();
    int t = 0;
    if (L.lane == 0) t = atomicAdd(a.tickets + wa, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t != (int)(wb - wa)) return;
    __threadfence();
    SmState<NC> m;
    m.reset();
    for (int64_t k = wa; k <= wb; ++k) {
        const float *sk = a.slots + (2 * k + (k == wa ? 1 : 0)) * stride;
        const float mk = L.active ? __ldcg(sk + a.HD + 2 * L.head) : -INFINITY;
        const float sk_s = L.active ? __ldcg(sk + a.HD + 2 * L.head + 1) : 0.f;
        const float mx = fmaxf(m.m, mk);
        const float c_old = (m.m == -INFINITY) ? 0.f : exp2f(m.m - mx);
        const float c_new = (mk == -INFINITY) ? 0.f : exp2f(mk - mx);
        m.s = m.s * c_old + sk_s * c_new;
        if (L.active) {
#pragma unroll
            for (int q = 0; q < NC; q += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(sk + L.lane * NC + q));
                m.acc[q] = m.acc[q] * c_old + v.x * c_new;
                m.acc[q + 1] = m.acc[q + 1] * c_old + v.y * c_new;
                m.acc[q + 2] = m.acc[q + 2] * c_old + v.z * c_new;
                m.acc[q + 3] = m.acc[q + 3] * c_old + v.w * c_new;
            }
        }
        m.m = mx;
    }
    store_final<KIND, T, CPL>(a, L, r, m);
    __syncwarp();
    if (L.lane == 0) a.tickets[wa] = 0;
}

// First row r with rowptr[r] >= e (binary search by lane 0, broadcast).
__device__ __forceinline__ int32_t warp_lower_bound(const int32_t *__restrict__ rowptr, int32_t n_rows,
                                                    int64_t e) {
    int32_t lo = 0;
    if ((threadIdx.x & 31) == 0) {
        int32_t hi = n_rows;
        while (lo < hi) {
            const int32_t mid = (lo + hi) >> 1;
            if ((int64_t)__ldg(rowptr + mid) < e) lo = mid + 1; else hi = mid;
        }
    }
    return __shfl_sync(0xffffffffu, lo, 0);
}

template <int KIND, class T, int CPL>
__global__ void __launch_bounds__(256) k_attn(AttnArgs a) {
    constexpr int NC = CPL * Elt<T>::N;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= a.n_workers) return;
    AttnLane<KIND, T, CPL> L;
    L.lane = threadIdx.x & 31;
    L.active = L.lane * CPL < a.nch;
    L.lph = a.D / NC;
    L.head = L.active ? (L.lane * NC) / a.D : 0;
    if (KIND == ATT_GATV2) {
#pragma unroll
        for (int k = 0; k < NC; ++k) L.coef[k] = L.active ? __ldg(a.coef + L.lane * NC + k) : 0.f;
    }
    const int64_t E = kAttnE;
    const int64_t e0 = w * E;
    const int64_t e1 = min(e0 + E, a.nnz);
    const int32_t *__restrict__ rowptr = a.rowptr;
    int32_t lo, lo_end;
    if (a.run_table) {
        lo = __ldg(a.run_table + w * kAttnRunMul);
        lo_end = (w + 1 == a.n_workers) ? a.n_rows : __ldg(a.run_table + (w + 1) * kAttnRunMul);
    } else {
        lo = warp_lower_bound(rowptr, a.n_rows, e0);
        lo_end = (w + 1 == a.n_workers) ? a.n_rows : warp_lower_bound(rowptr, a.n_rows, e1);
    }
    float dq[NC];
    float al;
    SmState<NC> st;
    // a heavy row that started in an earlier run and reaches into this one
    if (lo > 0 && e0 < a.nnz) {
        const int32_t lo_beg = __ldg(rowptr + lo);
        if (lo_beg > e0) {
            const int32_t h = lo - 1;
            if (lo_beg - __ldg(rowptr + h) > E) {
                load_dest<KIND, T, CPL>(a, L, h, dq, &al);
                st.reset();
                attend_range<KIND, T, CPL>(a, L, (int32_t)e0, (int32_t)min((int64_t)lo_beg, e1), dq, al, st);
                flush_piece<KIND, T, CPL>(a, L, w, h, st);
            }
        }
    }
    for (int32_t r = lo; r < lo_end; ++r) {
        const int32_t rb = __ldg(rowptr + r), re = __ldg(rowptr + r + 1);
        st.reset();
        if (re == rb) {
            store_final<KIND, T, CPL>(a, L, r, st);
            continue;
        }
        load_dest<KIND, T, CPL>(a, L, r, dq, &al);
        if (re - rb > E) {  // heavy: this run holds its first piece (and it is the last owned row)
            attend_range<KIND, T, CPL>(a, L, rb, (int32_t)e1, dq, al, st);
            flush_piece<KIND, T, CPL>(a, L, w, r, st);
        } else {
            attend_range<KIND, T, CPL>(a, L, rb, re, dq, al, st);
            store_final<KIND, T, CPL>(a, L, r, st);
        }
    }
}

// GATv2 per-node linear parts: A[i,h] = log2e * sum_d a'_hd C[i, hD+d] with
// a' = (1+s)/2 a.  One warp per node; lanes stride over the channels.
template <class T>
__global__ void __launch_bounds__(256) k_gatv2_linear(const T *__restrict__ C, int64_t n, int32_t heads,
                                                      int32_t D, const float *__restrict__ a,
                                                      float half_1ps, float *__restrict__ A) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= n) return;
    for (int32_t h = 0; h < heads; ++h) {
        float s = 0.f;
        for (int32_t d = lane; d < D; d += 32) {
            float c;
            if constexpr (sizeof(T) == 4) c = (float)C[i * heads * D + h * D + d];
            else c = __bfloat162float(C[i * heads * D + h * D + d]);
            s = fmaf(__ldg(a + h * D + d), c, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) A[i * heads + h] = s * half_1ps * kLog2e;
    }
}

// coef[c] = (1-s)/2 a[c] log2e (the |.| part), lin[c] = (1+s)/2 a[c] log2e
// (the linear part)
__global__ void k_gatv2_coef(const float *__restrict__ a, int32_t HD, float half_1ms, float half_1ps,
                             float *__restrict__ coef, float *__restrict__ lin) {
    const int32_t c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c < HD) {
        coef[c] = a[c] * half_1ms * kLog2e;
        lin[c] = a[c] * half_1ps * kLog2e;
    }
}

// ---------------------------------------------------------------- SIMT GEMM
// C[n, Fo] = H[n, Fi] W[Fi, Fo], fp32 FMA (no TF32), output in T (bf16 by
// round-to-nearest-even).  64x64 tile per 256-thread block, 4x4 per thread.
template <class T>
__global__ void __launch_bounds__(256) k_proj_simt(const T *__restrict__ H, const T *__restrict__ W,
                                                   T *__restrict__ C, int64_t n, int32_t Fi,
                                                   int32_t Fo) {
    __shared__ float sH[16][64 + 4];
    __shared__ float sW[16][64 + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int64_t row0 = (int64_t)blockIdx.x * 64;
    const int32_t col0 = blockIdx.y * 64;
    float acc[4][4] = {};
    auto ld = [](const T *p) -> float {
        if constexpr (sizeof(T) == 4) return (float)*p;
        else return __bfloat162float(*p);
    };
    for (int32_t k0 = 0; k0 < Fi; k0 += 16) {
        for (int t = threadIdx.x; t < 16 * 64; t += 256) {
            const int kk = t / 64, rr = t % 64;
            const int64_t gr = row0 + rr;
            sH[kk][rr] = (gr < n && k0 + kk < Fi) ? ld(H + gr * Fi + k0 + kk) : 0.f;
            const int32_t gc = col0 + rr;
            sW[kk][rr] = (gc < Fo && k0 + kk < Fi) ? ld(W + (int64_t)(k0 + kk) * Fo + gc) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float hv[4], wv[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                hv[q] = sH[kk][ty * 4 + q];
                wv[q] = sW[kk][tx * 4 + q];
            }
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(hv[p], wv[q], acc[p][q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int64_t gr = row0 + ty * 4 + p;
        if (gr >= n) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int32_t gc = col0 + tx * 4 + q;
            if (gc >= Fo) continue;
            if constexpr (sizeof(T) == 4) C[gr * Fo + gc] = acc[p][q];
            else C[gr * Fo + gc] = __float2bfloat16_rn(acc[p][q]);
        }
    }
}

}  // namespace

// tcgen05 projection (bf16), defined in projection.cu; returns
// GNN_ERR_UNSUPPORTED for shapes it does not cover.
gnn_status projection_tc(const void *H, int64_t n, int32_t F_in, const void *W, int32_t F_out,
                         void *C, cudaStream_t s);
gnn_status projection_tc_lin(const void *H, int64_t n, int32_t Fi, const void *W, int32_t Fo, void *C,
                             const float *lin_coef, int32_t heads, int32_t D, float *lin_out, cudaStream_t s);

static gnn_status projection_any(const void *H, int32_t dtype, int64_t n, int32_t F_in, const void *W,
                                 int32_t F_out, void *C, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    if (dtype == GNN_BF16) {
        gnn_status st = projection_tc(H, n, F_in, W, F_out, C, s);
        if (st != GNN_ERR_UNSUPPORTED) return st;
    }
    dim3 grid((unsigned)((n + 63) / 64), (unsigned)((F_out + 63) / 64));
    if (dtype == GNN_F32)
        k_proj_simt<float><<<grid, 256, 0, s>>>(static_cast<const float *>(H), static_cast<const float *>(W),
                                                 static_cast<float *>(C), n, F_in, F_out);
    else
        k_proj_simt<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(H),
                                                         static_cast<const __nv_bfloat16 *>(W),
                                                         static_cast<__nv_bfloat16 *>(C), n, F_in, F_out);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

static int64_t attn_workers(const gnn_csr *g) { return n_runs(g->nnz, kAttnE); }

static size_t attn_slot_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim) {
    const int64_t nw = attn_workers(g);
    return round_up(sizeof(float) * (size_t)2 * nw * (size_t)slot_stride(heads * head_dim, heads), 256) +
           round_up(sizeof(int32_t) * (size_t)nw, 256);
}

struct GatLayout {
    void *l, *r;
    float *Al, *Ar, *coef, *lin, *slots;
    int32_t *tickets;
    size_t bytes;
};

static GatLayout gat_layout(const gnn_csr *g, void *base, int32_t esize, bool separate, int32_t heads,
                            int32_t head_dim) {
    Carver c(base);
    GatLayout L;
    const size_t HD = (size_t)heads * head_dim;
    const int64_t nw = attn_workers(g);
    L.l = c.take<char>((size_t)g->n_cols * HD * esize);
    L.r = separate ? c.take<char>((size_t)g->n_cols * HD * esize) : L.l;
    L.Al = c.take<float>((size_t)g->n_cols * heads);
    L.Ar = separate ? c.take<float>((size_t)g->n_cols * heads) : L.Al;
    L.coef = c.take<float>(HD);
    L.lin = c.take<float>(HD);
    L.slots = c.take<float>((size_t)2 * nw * (size_t)slot_stride((int32_t)HD, heads));
    L.tickets = c.take<int32_t>((size_t)nw);
    L.bytes = c.used;
    return L;
}

size_t gatv2_workspace_bytes(const gnn_csr *g, int32_t F_in, int32_t heads, int32_t head_dim,
                             int32_t esize) {
    (void)F_in;
    // sized for separate W_l / W_r (the larger case)
    return gat_layout(g, nullptr, esize, true, heads, head_dim).bytes;
}

size_t gt_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim) {
    return attn_slot_bytes(g, heads, head_dim);
}

template <int KIND, class T>
static void launch_attn(const AttnArgs &a, int cpl, cudaStream_t s) {
    const int64_t threads = a.n_workers * 32;
    const int blocks = (int)((threads + 255) / 256);
    if constexpr (sizeof(T) == 2) {
        k_attn<KIND, T, 1><<<blocks, 256, 0, s>>>(a);  // bf16: at most 256 channels
    } else {
        switch (cpl) {
            case 1: k_attn<KIND, T, 1><<<blocks, 256, 0, s>>>(a); break;
            case 2: k_attn<KIND, T, 2><<<blocks, 256, 0, s>>>(a); break;
            case 4: k_attn<KIND, T, 4><<<blocks, 256, 0, s>>>(a); break;
            default: k_attn<KIND, T, 8><<<blocks, 256, 0, s>>>(a); break;
        }
    }
}

// Lane layout for HD channels of dtype; false if unsupported.
static bool attn_shape(int32_t dtype, int32_t heads, int32_t head_dim, int32_t *nch, int32_t *cpl) {
    const int nv = dtype == GNN_F32 ? 4 : 8;
    if (heads <= 0 || (head_dim != 32 && head_dim != 64 && head_dim != 128)) return false;
    const int32_t HD = heads * head_dim;
    if (HD % nv) return false;
    const int32_t ch = HD / nv;
    int32_t c = 1;
    while (ch > 32 * c) c *= 2;
    if (c > (dtype == GNN_F32 ? 8 : 1) || ch % c) return false;
    if (head_dim % (c * nv)) return false;  // a lane's channels must lie in one head
    *nch = ch;
    *cpl = c;
    return true;
}

// tensor-core tile path of GT attention over a block-sparse layout (tiles.cu)
gnn_status gt_attn_tiles(const gnn_csr *g, const gnn_blocksparse *bs, const void *Q, const void *K,
                         const void *V, int32_t heads, int32_t head_dim, float scale, float *out,
                         float *lse, void *ws, size_t ws_bytes, cudaStream_t s);

}  // namespace gnn

using namespace gnn;

extern "C" {

gnn_status gnn_projection(const void *H, int32_t dtype, int64_t n, int32_t F_in, const void *W,
                          int32_t F_out, void *C, void *stream) {
    if (n < 0 || F_in <= 0 || F_out <= 0) return GNN_ERR_INVALID_ARG;
    if (dtype != GNN_F32 && dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    if (n > 0 && (!H || !W || !C)) return GNN_ERR_INVALID_ARG;
    return projection_any(H, dtype, n, F_in, W, F_out, C, as_stream(stream));
}

gnn_status gnn_gatv2_fwd(const gnn_csr *g, const void *prep, const void *H, int32_t dtype,
                         int32_t F_in, const void *W_l, const void *W_r, const float *a,
                         int32_t heads, int32_t head_dim, float neg_slope, float *out,
                         float *lse, void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols) return GNN_ERR_UNSUPPORTED;
    if (dtype != GNN_F32 && dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    int32_t nch = 0, cpl = 0;
    if (!attn_shape(dtype, heads, head_dim, &nch, &cpl)) return GNN_ERR_UNSUPPORTED;
    if (F_in <= 0) return GNN_ERR_INVALID_ARG;
    if (!out || !a || !W_l || (!H && g->n_rows > 0)) return GNN_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(H)) return GNN_ERR_INVALID_ARG;
    if (g->n_rows == 0) return GNN_OK;
    const int32_t esize = dtype == GNN_F32 ? 4 : 2;
    const bool separate = W_r != nullptr;
    GatLayout WL = gat_layout(g, ws, esize, separate, heads, head_dim);
    if (!ws || ws_bytes < WL.bytes) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    cudaStream_t s = as_stream(stream);
    const int32_t HD = heads * head_dim;
    const int64_t n = g->n_cols;

    // coefficients of the |.| part and of the per-node linear parts
    const float half_1ps = 0.5f * (1.f + neg_slope), half_1ms = 0.5f * (1.f - neg_slope);
    k_gatv2_coef<<<(HD + 255) / 256, 256, 0, s>>>(a, HD, half_1ms, half_1ps, WL.coef, WL.lin);
    note_launch();
    GNN_LAUNCH_CHECK();
    // a3: projections l = H W_l (and r = H W_r) with the linear parts A_l, A_r
    const void *Ws[2] = {W_l, W_r};
    void *Cs[2] = {WL.l, WL.r};
    float *As[2] = {WL.Al, WL.Ar};
    for (int k = 0; k < (separate ? 2 : 1); ++k) {
        st = GNN_ERR_UNSUPPORTED;
        if (dtype == GNN_BF16)
            st = projection_tc_lin(H, n, F_in, Ws[k], HD, Cs[k], WL.lin, heads, head_dim, As[k], s);
        if (st == GNN_ERR_UNSUPPORTED) {
            st = projection_any(H, dtype, n, F_in, Ws[k], HD, Cs[k], s);
            if (st != GNN_OK) return st;
            const int lin_blocks = (int)((n * 32 + 255) / 256);
            if (dtype == GNN_F32)
                k_gatv2_linear<float><<<lin_blocks, 256, 0, s>>>(static_cast<const float *>(Cs[k]), n, heads,
                                                                  head_dim, a, half_1ps, As[k]);
            else
                k_gatv2_linear<__nv_bfloat16><<<lin_blocks, 256, 0, s>>>(
                    static_cast<const __nv_bfloat16 *>(Cs[k]), n, heads, head_dim, a, half_1ps, As[k]);
            note_launch();
            GNN_LAUNCH_CHECK();
        } else if (st != GNN_OK) {
            return st;
        }
    }

    AttnArgs A{};
    A.rowptr = g->rowptr;
    A.colidx = g->colidx;
    A.run_table = prep ? prep_run_table(g, prep) : nullptr;
    A.Sg = static_cast<const uint4 *>(WL.r);
    A.Vg = A.Sg;
    A.Qd = static_cast<const uint4 *>(WL.l);
    A.Al = WL.Al;
    A.Ar = WL.Ar;
    A.coef = WL.coef;
    A.out = out;
    A.lse = lse;
    A.slots = WL.slots;
    A.tickets = WL.tickets;
    A.nnz = g->nnz;
    A.n_workers = attn_workers(g);
    A.n_rows = g->n_rows;
    A.HD = HD;
    A.heads = heads;
    A.D = head_dim;
    A.nch = nch;
    if (dtype == GNN_F32) launch_attn<ATT_GATV2, float>(A, cpl, s);
    else launch_attn<ATT_GATV2, __nv_bfloat16>(A, cpl, s);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

gnn_status gnn_gt_attn_fwd(const gnn_csr *g, const void *prep, const gnn_blocksparse *bs,
                           const void *Q, const void *K, const void *V, int32_t dtype,
                           int32_t heads, int32_t head_dim, float scale, float *out,
                           float *lse, void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols) return GNN_ERR_UNSUPPORTED;
    if (dtype != GNN_F32 && dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    int32_t nch = 0, cpl = 0;
    if (!attn_shape(dtype, heads, head_dim, &nch, &cpl)) return GNN_ERR_UNSUPPORTED;
    if (!out || (g->n_rows > 0 && (!Q || !K || !V))) return GNN_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(Q) || !aligned16(K) || !aligned16(V)) return GNN_ERR_INVALID_ARG;
    if (g->n_rows == 0) return GNN_OK;
    cudaStream_t s = as_stream(stream);
    if (bs) {
        if (dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
        return gt_attn_tiles(g, bs, Q, K, V, heads, head_dim, scale, out, lse, ws, ws_bytes, s);
    }
    const size_t need = attn_slot_bytes(g, heads, head_dim);
    if (!ws || ws_bytes < need) return GNN_ERR_WORKSPACE;
    if (!aligned256(ws)) return GNN_ERR_INVALID_ARG;
    Carver cv(ws);
    AttnArgs A{};
    A.rowptr = g->rowptr;
    A.colidx = g->colidx;
    A.run_table = prep ? prep_run_table(g, prep) : nullptr;
    A.Sg = static_cast<const uint4 *>(K);
    A.Vg = static_cast<const uint4 *>(V);
    A.Qd = static_cast<const uint4 *>(Q);
    A.qscale = scale * kLog2e;
    A.out = out;
    A.lse = lse;
    A.n_workers = attn_workers(g);
    A.slots = cv.take<float>((size_t)2 * A.n_workers * (size_t)slot_stride(heads * head_dim, heads));
    A.tickets = cv.take<int32_t>((size_t)A.n_workers);
    A.nnz = g->nnz;
    A.n_rows = g->n_rows;
    A.HD = heads * head_dim;
    A.heads = heads;
    A.D = head_dim;
    A.nch = nch;
    if (dtype == GNN_F32) launch_attn<ATT_GT, float>(A, cpl, s);
    else launch_attn<ATT_GT, __nv_bfloat16>(A, cpl, s);
    note_launch();
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

}  // extern "C"
