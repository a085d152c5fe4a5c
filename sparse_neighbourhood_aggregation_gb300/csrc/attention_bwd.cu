// Backward of the fused Graph Transformer attention.
//
// IO-aware GNN layers, Appendix D.2 (the GT backward: Delta = <O, dO> per
// destination and head in a kernel of its own, then the kernels over CSR and
// CSR^T that recompute the weights from the stored logsumexp L).  For row i,
// head h, edge j in N(i), with s_ij = scale <q_i, k_j>:
//   alpha_ij = exp(s_ij - L_i),  ds_ij = alpha_ij (<dO_i, v_j> - Delta_i)
//   dQ_i = scale sum_j ds_ij k_j          (over the CSR)
//   dK_j = scale sum_i ds_ij q_i,  dV_j = sum_i alpha_ij dO_i   (over CSR^T)
// Two schedules: a warp per row (k_gt_bwd_q, k_gt_bwd_kv) on graphs of long,
// even rows, and the GATv2 backward's edge runs (k_gt_bwd_run) on power-law
// graphs, chosen by the mean degree.
// Each gradient row is owned by one warp, so there are no atomics and the
// sums are deterministic.  Lane l holds channels [l*NC, (l+1)*NC) of the
// HD = 32 NC channels; the D / NC lanes of a head reduce its dot products
// with shuffles.  The edge loop loads the rows of U edges before using any.
//
// Backward of the fused GATv2 attention (same appendix, the GATv2 backward:
// an AL kernel for the left features and the attention vector, which also
// forms G_i = sum_j alpha_ij <dO_i, r_j>, and an R kernel over CSR^T for the
// right features; the attention-vector gradient is reduced over nodes at the
// end).  With x_ij = l_i + r_j per head, sigma = LeakyReLU(slope), e_ij =
// <a_h, sigma(x_ij)> and alpha_ij = exp(e_ij - L_i):
//   de_ij = alpha_ij (<dO_i, r_j> - G_i)
//   dl_i  = sum_j de_ij a_h . sigma'(x_ij)              (k_gatv2_bwd<AL>)
//   da_h  = sum_ij de_ij sigma(x_ij)                     (AL, then k_gatv2_bwd_da)
//   dr_j  = sum_i alpha_ij dO_i + de_ij a_h . sigma'(x_ij)  (k_gatv2_bwd<R>)
// G_i is formed as <O_i, dO_i>, the same number since O_i = sum_j alpha_ij
// r_j, so no pass over the row is spent on it before the gradients.
// Schedule: power-law graphs have rows of tens of thousands of edges, so a
// warp per row would leave one warp with a hub's whole list.  A warp is a
// worker over a run of kGatE consecutive edges instead (the forward's
// schedule): it owns the rows whose first edge lies in its run, processes a
// light row whole, and cuts a heavy row (degree > kGatE) at run boundaries.
// Every piece of a heavy row leaves its partial gradient row in a slot; the
// last piece to finish (ticket counter, no waiting) sums the slots in edge
// order, so the result does not depend on which warp ran first.  The
// attention-vector gradient is kept per warp in registers, summed per block,
// and the block partials are summed in a fixed order by k_gatv2_bwd_da.
#include <algorithm>

#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);

namespace {

// Edges whose rows a warp loads together.  One edge at a time is the
// fastest on a clustered 262K-node graph (8 heads x 32): 4.8 ms per
// backward, against 6.0-7.5 ms with 2, 7.5 with 4 and 13.7 with 8, and
// asking for more resident blocks made it slower still; the gathered rows
// thrash L1 before they are reused, so fewer rows in flight win.
#ifndef GNN_GT_BWD_U
#define GNN_GT_BWD_U 1
#endif
constexpr int kBwdU = GNN_GT_BWD_U;

struct GtBwdArgs {
    const int32_t *rowptr, *colidx;      // CSR (destination rows) or CSR^T (source rows)
    const __nv_bfloat16 *Q, *K, *V;
    const float *O, *lse, *dO;
    float *delta;                        // [n, heads]
    float *dA, *dB;                      // q kernel: dQ; kv kernel: dK, dV
    int32_t n, heads, D, HD;
    float scale;
};

template <int NC>
__device__ __forceinline__ void ld_bf16(const __nv_bfloat16 *p, float *f) {
    if constexpr (NC == 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
        f[0] = bf16lo(v.x); f[1] = bf16hi(v.x); f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    } else {
#pragma unroll
        for (int c = 0; c < NC / 8; ++c) {
            const uint4 v = ldg16(p + 8 * c);
            Chunk<__nv_bfloat16>::unpack(v, f + 8 * c);
        }
    }
}

template <int NC>
__device__ __forceinline__ void ld_f32(const float *p, float *f) {
#pragma unroll
    for (int c = 0; c < NC; c += 4) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(p + c));
        f[c] = v.x; f[c + 1] = v.y; f[c + 2] = v.z; f[c + 3] = v.w;
    }
}

template <int NC>
__device__ __forceinline__ void st_f32(float *p, const float *f) {
#pragma unroll
    for (int c = 0; c < NC; c += 4) *reinterpret_cast<float4 *>(p + c) = make_float4(f[c], f[c + 1], f[c + 2], f[c + 3]);
}

// sum over the lph lanes of this lane's head (lph a power of two).  LPH > 0
// fixes lph at compile time: the shuffles then unroll, where a loop with a
// runtime trip count makes the compiler guard every shuffle against
// divergence (measured on GB300 in the GATv2 backward: ~35 of its 210 warp
// instructions per edge were those guards)
template <int LPH>
__device__ __forceinline__ float head_sum(float x, int lph) {
    if constexpr (LPH > 0) {
#pragma unroll
        for (int o = LPH >> 1; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    } else {
        for (int o = lph >> 1; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    }
    return x;
}

template <int NC, int LPH>
__global__ void __launch_bounds__(256) k_gt_bwd_q(GtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int32_t i = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (i >= a.n) return;
    const int lph = LPH > 0 ? LPH : a.D / NC;
    const int h = (lane * NC) / a.D;
    const int64_t ro = (int64_t)i * a.HD + lane * NC;
    float q[NC], o[NC], g[NC], dq[NC];
    ld_bf16<NC>(a.Q + ro, q);
    ld_f32<NC>(a.O + ro, o);
    ld_f32<NC>(a.dO + ro, g);
    // Delta = <O_i, dO_i> in the same two-chain order as <dO_i, v_j> below,
    // so a row whose only edge gives O_i = v_j gets ds = 0 exactly
    uint64_t p2 = pk2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < NC; c += 2) p2 = fma2(pk2(g[c], g[c + 1]), pk2(o[c], o[c + 1]), p2);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        q[c] *= a.scale;
        dq[c] = 0.f;
    }
    float p0, p1;
    upk2(p2, p0, p1);
    const float delta = head_sum<LPH>(p0 + p1, lph);
    const int32_t b = __ldg(a.rowptr + i), e = __ldg(a.rowptr + i + 1);
    const float L = e > b ? __ldg(a.lse + (int64_t)i * a.heads + h) : 0.f;
    for (int32_t cb = b; cb < e; cb += 32) {
        const int32_t cj = cb + lane < e ? __ldg(a.colidx + cb + lane) : 0;
        const int n = min(32, e - cb);
        for (int u0 = 0; u0 < n; u0 += kBwdU) {
            float kf[kBwdU][NC], vf[kBwdU][NC];
#pragma unroll
            for (int u = 0; u < kBwdU; ++u) {
                const int32_t j = __shfl_sync(0xffffffffu, cj, (u0 + u) & 31);
                if (u0 + u < n) {
                    ld_bf16<NC>(a.K + (int64_t)j * a.HD + lane * NC, kf[u]);
                    ld_bf16<NC>(a.V + (int64_t)j * a.HD + lane * NC, vf[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < kBwdU; ++u) {
                if (u0 + u >= n) break;
                // <q_i, k_j> and <dO_i, v_j> on pairs of channels (f32x2)
                uint64_t s2 = pk2(0.f, 0.f), d2 = pk2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < NC; c += 2) {
                    s2 = fma2(pk2(q[c], q[c + 1]), pk2(kf[u][c], kf[u][c + 1]), s2);
                    d2 = fma2(pk2(g[c], g[c + 1]), pk2(vf[u][c], vf[u][c + 1]), d2);
                }
                float s0, s1, d0, d1;
                upk2(s2, s0, s1);
                upk2(d2, d0, d1);
                const float s = head_sum<LPH>(s0 + s1, lph);
                const float da = head_sum<LPH>(d0 + d1, lph);
                const float ds = __expf(s - L) * (da - delta);
                const uint64_t ds2 = pk2(ds, ds);
#pragma unroll
                for (int c = 0; c < NC; c += 2)
                    upk2(fma2(ds2, pk2(kf[u][c], kf[u][c + 1]), pk2(dq[c], dq[c + 1])), dq[c], dq[c + 1]);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) dq[c] *= a.scale;
    st_f32<NC>(a.dA + ro, dq);
    if (lane % lph == 0) a.delta[(int64_t)i * a.heads + h] = delta;
}

template <int NC, int LPH>
__global__ void __launch_bounds__(256) k_gt_bwd_kv(GtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int32_t j = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (j >= a.n) return;
    const int lph = LPH > 0 ? LPH : a.D / NC;
    const int h = (lane * NC) / a.D;
    const int64_t ro = (int64_t)j * a.HD + lane * NC;
    float kf[NC], vf[NC], dk[NC], dv[NC];
    ld_bf16<NC>(a.K + ro, kf);
    ld_bf16<NC>(a.V + ro, vf);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        kf[c] *= a.scale;
        dk[c] = 0.f;
        dv[c] = 0.f;
    }
    const int32_t b = __ldg(a.rowptr + j), e = __ldg(a.rowptr + j + 1);
    for (int32_t cb = b; cb < e; cb += 32) {
        const int32_t ci = cb + lane < e ? __ldg(a.colidx + cb + lane) : 0;
        const int n = min(32, e - cb);
        for (int u0 = 0; u0 < n; u0 += kBwdU) {
            float qf[kBwdU][NC], gf[kBwdU][NC], Lh[kBwdU], Dh[kBwdU];
#pragma unroll
            for (int u = 0; u < kBwdU; ++u) {
                const int32_t i = __shfl_sync(0xffffffffu, ci, (u0 + u) & 31);
                if (u0 + u < n) {
                    const int64_t io = (int64_t)i * a.HD + lane * NC;
                    ld_bf16<NC>(a.Q + io, qf[u]);
                    ld_f32<NC>(a.dO + io, gf[u]);
                    Lh[u] = __ldg(a.lse + (int64_t)i * a.heads + h);
                    Dh[u] = __ldg(a.delta + (int64_t)i * a.heads + h);
                }
            }
#pragma unroll
            for (int u = 0; u < kBwdU; ++u) {
                if (u0 + u >= n) break;
                uint64_t s2 = pk2(0.f, 0.f), d2 = pk2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < NC; c += 2) {
                    s2 = fma2(pk2(qf[u][c], qf[u][c + 1]), pk2(kf[c], kf[c + 1]), s2);
                    d2 = fma2(pk2(gf[u][c], gf[u][c + 1]), pk2(vf[c], vf[c + 1]), d2);
                }
                float s0, s1, d0, d1;
                upk2(s2, s0, s1);
                upk2(d2, d0, d1);
                const float s = head_sum<LPH>(s0 + s1, lph);
                const float da = head_sum<LPH>(d0 + d1, lph);
                const float al = __expf(s - Lh[u]);
                const float ds = al * (da - Dh[u]);
                const uint64_t al2 = pk2(al, al), ds2 = pk2(ds, ds);
#pragma unroll
                for (int c = 0; c < NC; c += 2) {
                    upk2(fma2(al2, pk2(gf[u][c], gf[u][c + 1]), pk2(dv[c], dv[c + 1])), dv[c], dv[c + 1]);
                    upk2(fma2(ds2, pk2(qf[u][c], qf[u][c + 1]), pk2(dk[c], dk[c + 1])), dk[c], dk[c + 1]);
                }
            }
        }
    }
    // the scale sits in k for the scores; dK = scale sum_i ds_ij q_i
#pragma unroll
    for (int c = 0; c < NC; ++c) dk[c] *= a.scale;
    st_f32<NC>(a.dA + ro, dk);
    st_f32<NC>(a.dB + ro, dv);
}

// ---------------------------------------------------------------- GATv2

constexpr int64_t kGatE = 256;     // edges per worker run
constexpr int kGatWarps = 8;       // warps per block
constexpr int kDaBlocks = 128;     // blocks of the attention-vector reduction

enum GatSide { GAT_AL = 0, GAT_R = 1 };

struct GatBwdArgs {
    const int32_t *rowptr, *colidx;  // AL: CSR (destination rows); R: CSR^T (source rows)
    const int32_t *run_rows;         // [n_runs + 1]: first row whose first edge is in run w
    const void *Cl, *Cr;             // l and r features [n, HD] (fp32 or bf16)
    const float *a;                  // [HD]
    const float *O, *lse, *dO;       // forward output, logsumexp [n, heads], grad of O
    float *G;                        // [n, heads]: AL writes, R reads
    float *grad;                     // AL: dl; R: dr  [n, HD]
    float *slots;                    // [2 n_runs, HD] partial rows of heavy-row pieces
    int32_t *tickets;                // [channel groups, n_runs], cleared at the start of a call
    float *da_part;                  // AL: [gridDim.x, HD] per-block attention-vector sums
    int64_t nnz, n_runs;
    int32_t n, heads, D, HD;
    float slope;
};

// NC channels of a feature row, widened to fp32
template <typename T, int NC>
__device__ __forceinline__ void ld_row(const void *base, int64_t off, float *f) {
    if constexpr (sizeof(T) == 4) {
        const float *p = static_cast<const float *>(base) + off;
        if constexpr (NC == 1) {
            f[0] = __ldg(p);
        } else if constexpr (NC == 2) {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
            f[0] = v.x; f[1] = v.y;
        } else {
#pragma unroll
            for (int c = 0; c < NC; c += 4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(p + c));
                f[c] = v.x; f[c + 1] = v.y; f[c + 2] = v.z; f[c + 3] = v.w;
            }
        }
    } else {
        const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + off;
        if constexpr (NC == 1) {
            f[0] = bf16lo(__ldg(reinterpret_cast<const unsigned short *>(p)));
        } else if constexpr (NC == 2) {
            const uint32_t v = __ldg(reinterpret_cast<const unsigned int *>(p));
            f[0] = bf16lo(v); f[1] = bf16hi(v);
        } else {
            ld_bf16<NC>(p, f);
        }
    }
}

template <int NC>
__device__ __forceinline__ void st_row(float *p, const float *f) {
    if constexpr (NC == 1) {
        *p = f[0];
    } else if constexpr (NC == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(f[0], f[1]);
    } else {
        st_f32<NC>(p, f);
    }
}

template <int NC>
__device__ __forceinline__ void st_row_cg(float *p, const float *f) {
#pragma unroll
    for (int c = 0; c < NC; ++c) __stcg(p + c, f[c]);
}

// Destination-side (AL) or source-side (R) data of the row a warp works on.
template <int SIDE, int NC>
struct GatRow {
    float own[NC];   // AL: l_i; R: r_j
    float g[NC];     // AL: dO_i
    float L, G;      // AL: logsumexp and G of (i, head)
};

template <int SIDE, typename T, int NC, int LPH>
__device__ __forceinline__ void gat_load_row(const GatBwdArgs &p, int32_t r, int ch, int hd, int lph,
                                             bool nonempty, GatRow<SIDE, NC> &R) {
    const int64_t ro = (int64_t)r * p.HD + ch;
    if constexpr (SIDE == GAT_AL) {
        ld_row<T, NC>(p.Cl, ro, R.own);
        float o[NC];
        ld_row<float, NC>(p.O, ro, o);
        ld_row<float, NC>(p.dO, ro, R.g);
        // G = <O_i, dO_i> in the order the edge loop forms <dO_i, r_j> (two
        // chains of channel pairs), so a row whose only edge gives O_i = r_j
        // gets de = 0 exactly
        float s = 0.f;
        if constexpr (NC == 1) {
            s = R.g[0] * o[0];
        } else {
            uint64_t s2 = pk2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < NC; c += 2) s2 = fma2(pk2(R.g[c], R.g[c + 1]), pk2(o[c], o[c + 1]), s2);
            float s0, s1;
            upk2(s2, s0, s1);
            s = s0 + s1;
        }
        R.G = head_sum<LPH>(s, lph);
        R.L = nonempty ? __ldg(p.lse + (int64_t)r * p.heads + hd) : 0.f;
    } else {
        ld_row<T, NC>(p.Cr, ro, R.own);
    }
}

// NC channels of a feature row as loaded (fp32, or bf16 words kept packed
// until use, so a load issued for the next edge is not waited on now).
template <typename T, int NC>
struct Raw {
    float f[NC];
    __device__ __forceinline__ void load(const void *base, int64_t off) {
        ld_row<float, NC>(base, off, f);
    }
    __device__ __forceinline__ void unpack(float *o) const {
#pragma unroll
        for (int c = 0; c < NC; ++c) o[c] = f[c];
    }
};

template <int NC>
struct Raw<__nv_bfloat16, NC> {
    uint32_t w[(NC + 1) / 2];
    __device__ __forceinline__ void load(const void *base, int64_t off) {
        const __nv_bfloat16 *p = static_cast<const __nv_bfloat16 *>(base) + off;
        if constexpr (NC == 1) {
            w[0] = __ldg(reinterpret_cast<const unsigned short *>(p));
        } else if constexpr (NC == 2) {
            w[0] = __ldg(reinterpret_cast<const unsigned int *>(p));
        } else if constexpr (NC == 4) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
            w[0] = v.x; w[1] = v.y;
        } else {
#pragma unroll
            for (int c = 0; c < NC / 8; ++c) {
                const uint4 v = ldg16(p + 8 * c);
                w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
            }
        }
    }
    __device__ __forceinline__ void unpack(float *o) const {
        if constexpr (NC == 1) {
            o[0] = bf16lo(w[0]);
        } else {
#pragma unroll
            for (int c = 0; c < NC / 2; ++c) { o[2 * c] = bf16lo(w[c]); o[2 * c + 1] = bf16hi(w[c]); }
        }
    }
};

// What one edge gathers: AL the neighbour's r_j; R the destination's l_i,
// dO_i, logsumexp and G.
template <int SIDE, typename T, int NC>
struct EdgeData {
    Raw<T, NC> v;
    Raw<float, NC> g;
    float L, G;
    __device__ __forceinline__ void load(const GatBwdArgs &p, int32_t k, int ch, int hd) {
        const int64_t ko = (int64_t)k * p.HD + ch;
        if constexpr (SIDE == GAT_AL) {
            v.load(p.Cr, ko);
        } else {
            v.load(p.Cl, ko);
            g.load(p.dO, ko);
            L = __ldg(p.lse + (int64_t)k * p.heads + hd);
            G = __ldg(p.G + (int64_t)k * p.heads + hd);
        }
    }
};

// Gradient contributions of the edges [eb, ee) of one row into acc (dl_i or
// dr_j) and, on the AL side, ga (attention vector).  The gathers run one
// edge ahead of the arithmetic.
template <int SIDE, typename T, int NC, int LPH>
__device__ __forceinline__ void gat_edges(const GatBwdArgs &p, const GatRow<SIDE, NC> &R, const float *av,
                                          int lane, int ch, int hd, int lph, int32_t eb, int32_t ee,
                                          float *acc, float *ga) {
    if (eb >= ee) return;
    int32_t base = eb;
    int32_t cn = base + lane < ee ? __ldg(p.colidx + base + lane) : 0;
    EdgeData<SIDE, T, NC> nxt;
    nxt.load(p, __shfl_sync(0xffffffffu, cn, 0), ch, hd);
    for (int32_t e = eb; e < ee; ++e) {
        const EdgeData<SIDE, T, NC> cur = nxt;
        if (e + 1 < ee) {
            if (e + 1 - base == 32) {
                base = e + 1;
                cn = base + lane < ee ? __ldg(p.colidx + base + lane) : 0;
            }
            nxt.load(p, __shfl_sync(0xffffffffu, cn, e + 1 - base), ch, hd);
        }
        float x[NC], rr[NC], gg[NC];
        float L, G;
        if constexpr (SIDE == GAT_AL) {
            cur.v.unpack(rr);                    // r_j of neighbour j
#pragma unroll
            for (int c = 0; c < NC; ++c) gg[c] = R.g[c];
            L = R.L;
            G = R.G;
        } else {
            cur.v.unpack(x);                     // l_i of destination i (x = l_i + r_j below)
            cur.g.unpack(gg);                    // dO_i
            L = cur.L;
            G = cur.G;
#pragma unroll
            for (int c = 0; c < NC; ++c) rr[c] = R.own[c];
        }
        // x = l_i + r_j; lr = LeakyReLU(x); the score and <dO_i, r_j> on
        // pairs of channels (f32x2), two chains each
        float lr[NC];
        uint64_t ev2 = pk2(0.f, 0.f), pr2 = pk2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
            if constexpr (NC == 1) {
                x[0] = (SIDE == GAT_AL ? R.own[0] : x[0]) + rr[0];
                lr[0] = x[0] > 0.f ? x[0] : p.slope * x[0];
                ev2 = pk2(av[0] * lr[0], 0.f);
                pr2 = pk2(gg[0] * rr[0], 0.f);
            } else {
                const uint64_t a2 = SIDE == GAT_AL ? pk2(R.own[c], R.own[c + 1]) : pk2(x[c], x[c + 1]);
                upk2(add2(a2, pk2(rr[c], rr[c + 1])), x[c], x[c + 1]);
                lr[c] = x[c] > 0.f ? x[c] : p.slope * x[c];
                lr[c + 1] = x[c + 1] > 0.f ? x[c + 1] : p.slope * x[c + 1];
                ev2 = fma2(pk2(av[c], av[c + 1]), pk2(lr[c], lr[c + 1]), ev2);
                pr2 = fma2(pk2(gg[c], gg[c + 1]), pk2(rr[c], rr[c + 1]), pr2);
            }
        }
        float e0, e1, p0, p1;
        upk2(ev2, e0, e1);
        upk2(pr2, p0, p1);
        const float ev = head_sum<LPH>(e0 + e1, lph);
        const float pr = head_sum<LPH>(p0 + p1, lph);
        const float al = __expf(ev - L);
        const float de = al * (pr - G);
        // sigma'(x) a = a or slope a, so de sigma'(x) is de or de slope; and
        // sigma'(x) x is LeakyReLU(x), already at hand
        const float ds = de * p.slope;
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
            if constexpr (NC == 1) {
                const float d = x[0] > 0.f ? de : ds;
                if constexpr (SIDE == GAT_AL) {
                    acc[0] = fmaf(d, av[0], acc[0]);
                    ga[0] = fmaf(de, lr[0], ga[0]);
                } else {
                    acc[0] = fmaf(al, gg[0], fmaf(d, av[0], acc[0]));
                }
            } else {
                const uint64_t d2 = pk2(x[c] > 0.f ? de : ds, x[c + 1] > 0.f ? de : ds);
                uint64_t a2 = fma2(d2, pk2(av[c], av[c + 1]), pk2(acc[c], acc[c + 1]));
                if constexpr (SIDE == GAT_AL) {
                    upk2(fma2(pk2(de, de), pk2(lr[c], lr[c + 1]), pk2(ga[c], ga[c + 1])), ga[c], ga[c + 1]);
                } else {
                    a2 = fma2(pk2(al, al), pk2(gg[c], gg[c + 1]), a2);
                }
                upk2(a2, acc[c], acc[c + 1]);
            }
        }
    }
}

// A piece of heavy row r leaves acc in its slot; the last of the row's
// pieces to arrive sums them in edge order and writes the gradient row.
template <int NC>
__device__ __forceinline__ void gat_flush_piece(const GatBwdArgs &p, int64_t w, int32_t r, int lane, int ch,
                                                const float *acc) {
    const int32_t rb = __ldg(p.rowptr + r), re = __ldg(p.rowptr + r + 1);
    const int64_t wa = rb / kGatE, wb = ((int64_t)re - 1) / kGatE;
    int32_t *ticket = p.tickets + blockIdx.y * p.n_runs + wa;  // one ticket set per channel group
    st_row_cg<NC>(p.slots + (2 * w + (w == wa ? 1 : 0)) * p.HD + ch, acc);
    __threadfence();
    __syncwarp();
    int t = 0;
    if (lane == 0) t = atomicAdd(ticket, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t != (int)(wb - wa)) return;
    __threadfence();
    float sum[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) sum[c] = 0.f;
    for (int64_t k = wa; k <= wb; ++k) {
        const float *sk = p.slots + (2 * k + (k == wa ? 1 : 0)) * p.HD + ch;
#pragma unroll
        for (int c = 0; c < NC; ++c) sum[c] += __ldcg(sk + c);
    }
    st_row<NC>(p.grad + (int64_t)r * p.HD + ch, sum);
    __syncwarp();
    if (lane == 0) *ticket = 0;
}

// Three resident blocks per SM (80 registers a thread): 9.3 ms for the
// whole backward on R-MAT scale 20 (4 heads x 64, bf16) against 11.4 ms at
// the compiler's 94 registers; the edge loop waits on gathers, so resident
// warps matter more than the few values spilled.
constexpr int kGatMinBlocks = 3;
template <int SIDE, typename T, int NC, int LPH>
__global__ void __launch_bounds__(kGatWarps * 32, kGatMinBlocks) k_gatv2_bwd(GatBwdArgs p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w = (int64_t)blockIdx.x * kGatWarps + warp;
    const int lph = LPH > 0 ? LPH : p.D / NC;
    const int ch = (int)blockIdx.y * 32 * NC + lane * NC;  // this lane's first channel
    const int hd = ch / p.D;
    float av[NC], ga[NC];
    ld_row<float, NC>(p.a, ch, av);
#pragma unroll
    for (int c = 0; c < NC; ++c) ga[c] = 0.f;
    if (w < p.n_runs) {
        const int64_t e0 = w * kGatE, e1 = min(e0 + kGatE, p.nnz);
        const int32_t lo = __ldg(p.run_rows + w), lo_end = __ldg(p.run_rows + w + 1);
        // a heavy row that started in an earlier run and reaches into this one
        if (lo > 0 && e0 < p.nnz) {
            const int32_t lo_beg = __ldg(p.rowptr + lo);
            if (lo_beg > e0 && lo_beg - __ldg(p.rowptr + lo - 1) > kGatE) {
                GatRow<SIDE, NC> R;
                gat_load_row<SIDE, T, NC, LPH>(p, lo - 1, ch, hd, lph, true, R);
                float acc[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[c] = 0.f;
                gat_edges<SIDE, T, NC, LPH>(p, R, av, lane, ch, hd, lph, (int32_t)e0,
                                       (int32_t)min((int64_t)lo_beg, e1), acc, ga);
                gat_flush_piece<NC>(p, w, lo - 1, lane, ch, acc);
            }
        }
        // owned rows, bounds read 32 at a time
        for (int32_t rbase = lo; rbase < lo_end; rbase += 32) {
            const int32_t rr = rbase + lane;
            int32_t my_b = 0, my_e = 0;
            if (rr < lo_end) {
                my_b = __ldg(p.rowptr + rr);
                my_e = __ldg(p.rowptr + rr + 1);
            }
            const int cnt = min(32, lo_end - rbase);
            for (int k = 0; k < cnt; ++k) {
                const int32_t r = rbase + k;
                const int32_t rb = __shfl_sync(0xffffffffu, my_b, k), re = __shfl_sync(0xffffffffu, my_e, k);
                GatRow<SIDE, NC> R;
                gat_load_row<SIDE, T, NC, LPH>(p, r, ch, hd, lph, re > rb, R);
                if constexpr (SIDE == GAT_AL) {
                    if (lane % lph == 0) p.G[(int64_t)r * p.heads + hd] = R.G;
                }
                float acc[NC];
#pragma unroll
                for (int c = 0; c < NC; ++c) acc[c] = 0.f;
                if (re - rb > kGatE) {  // heavy: its first piece (the last owned row)
                    gat_edges<SIDE, T, NC, LPH>(p, R, av, lane, ch, hd, lph, rb, (int32_t)e1, acc, ga);
                    gat_flush_piece<NC>(p, w, r, lane, ch, acc);
                } else {
                    gat_edges<SIDE, T, NC, LPH>(p, R, av, lane, ch, hd, lph, rb, re, acc, ga);
                    st_row<NC>(p.grad + (int64_t)r * p.HD + ch, acc);
                }
            }
        }
    }
    if constexpr (SIDE == GAT_AL) {
        // per-block sum of the warps' attention-vector gradients over this
        // block's channel group, in warp order
        __shared__ float sga[kGatWarps][32 * NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) sga[warp][lane * NC + c] = ga[c];
        __syncthreads();
        for (int c = threadIdx.x; c < 32 * NC; c += blockDim.x) {
            float t = 0.f;
#pragma unroll
            for (int k = 0; k < kGatWarps; ++k) t += sga[k][c];
            p.da_part[(int64_t)blockIdx.x * p.HD + blockIdx.y * 32 * NC + c] = t;
        }
    }
}

// run_rows[w] = first row r with rowptr[r] >= w * kGatE, for the runs of the
// CSR (run_rows) and of CSR^T (run_rows_t); run_rows[n_runs] = n.  Thread r
// (0 <= r <= n) covers the runs whose start lies in (rowptr[r-1], rowptr[r]];
// r = n takes the runs that start inside the last row (no row begins there).
// Also clears the tickets (every channel group's) and the reduction ticket.
__global__ void k_gatv2_bwd_runs(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ rowptr_t,
                                 int32_t n, int64_t n_runs, int32_t *__restrict__ run_rows,
                                 int32_t *__restrict__ run_rows_t, int32_t *__restrict__ tickets,
                                 int64_t n_tickets, int32_t *__restrict__ da_ticket) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t t = r; t < n_tickets; t += (int64_t)gridDim.x * blockDim.x) tickets[t] = 0;
    if (r == 0) *da_ticket = 0;
    if (r > n) return;
    if (r == n) {
        run_rows[n_runs] = n;
        run_rows_t[n_runs] = n;
    }
    const int32_t *rps[2] = {rowptr, rowptr_t};
    int32_t *outs[2] = {run_rows, run_rows_t};
    for (int k = 0; k < 2; ++k) {
        const int64_t hi = rps[k][r];
        const int64_t lo = r > 0 ? (int64_t)rps[k][r - 1] + 1 : 0;
        for (int64_t w = (lo + kGatE - 1) / kGatE; w * kGatE <= hi && w < n_runs; ++w) outs[k][w] = (int32_t)r;
    }
}

// da[c] = sum over the AL blocks of da_part[b, c]: block q sums a fixed
// slice of the partial rows, the last block to finish sums the slices in
// order.
__global__ void __launch_bounds__(256) k_gatv2_bwd_da(const float *__restrict__ part, int64_t n_part, int32_t HD,
                                                      float *__restrict__ part2, int32_t *__restrict__ ticket,
                                                      float *__restrict__ da) {
    const int c = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * n_part / gridDim.x;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * n_part / gridDim.x;
    if (c < HD) {
        float s = 0.f;
        for (int64_t r = r0; r < r1; ++r) s += __ldg(part + r * HD + c);
        __stcg(part2 + (int64_t)blockIdx.x * HD + c, s);
    }
    __threadfence();
    __syncthreads();
    __shared__ int last;
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (c < HD) {
        float t = 0.f;
        for (int q = 0; q < (int)gridDim.x; ++q) t += __ldcg(part2 + (int64_t)q * HD + c);
        da[c] = t;
    }
    if (threadIdx.x == 0) *ticket = 0;
}

// ---------------------------------------------------------------- GT on edge runs

// The GT backward on the GATv2 backward's schedule: a warp per run of kGatE
// edges, owning the rows whose first edge lies in its run, a heavy row cut at
// run boundaries and its pieces summed in edge order by the last to finish.
// Q side over CSR (rows = destinations i): Delta_i = <O_i, dO_i>, then for
// every edge j: s = <q_i, k_j> scale, alpha = exp(s - L_i), ds = alpha
// (<dO_i, v_j> - Delta_i), dQ_i += scale ds k_j.  KV side over CSR^T (rows
// = sources j): for every edge i: dV_j += alpha dO_i, dK_j += scale ds q_i.
// Delta_i is formed by every warp that holds a piece of row i (a few
// multiply-adds) and stored by the row's owner for the KV side.
enum GtSide { GT_Q = 0, GT_KV = 1 };

struct GtRunArgs {
    const int32_t *rowptr, *colidx;  // Q: CSR; KV: CSR^T
    const int32_t *run_rows;         // [n_runs + 1]
    const __nv_bfloat16 *Q, *K, *V;
    const float *O, *lse, *dO;
    float *delta;                    // [n, heads]: Q writes, KV reads
    float *dA, *dB;                  // Q: dQ; KV: dK, dV  [n, HD]
    float *slots;                    // [2 n_runs, 2 HD] partial rows of heavy-row pieces
    int32_t *tickets;                // [n_runs], zero on entry and on exit
    int64_t nnz, n_runs;
    int32_t n, heads, D, HD;
    float scale;
};

// The row-side data of row r: Q side q_i (scaled), dO_i, L_i, Delta_i;
// KV side k_j (scaled) and v_j.
template <int SIDE, int NC, int LPH>
struct GtRow {
    float a[NC], b[NC];  // Q: q, dO;  KV: k, v
    float L, Dl;
    __device__ __forceinline__ void load(const GtRunArgs &p, int32_t r, int ch, int hd, int lph, bool nonempty) {
        const int64_t ro = (int64_t)r * p.HD + ch;
        if constexpr (SIDE == GT_Q) {
            ld_bf16<NC>(p.Q + ro, a);
            float o[NC];
            ld_f32<NC>(p.O + ro, o);
            ld_f32<NC>(p.dO + ro, b);
            // Delta in the two-chain order of <dO_i, v_j> below: a row whose
            // only edge gives O_i = v_j gets ds = 0 exactly
            uint64_t p2 = pk2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < NC; c += 2) p2 = fma2(pk2(b[c], b[c + 1]), pk2(o[c], o[c + 1]), p2);
            float p0, p1;
            upk2(p2, p0, p1);
            Dl = head_sum<LPH>(p0 + p1, lph);
            L = nonempty ? __ldg(p.lse + (int64_t)r * p.heads + hd) : 0.f;
#pragma unroll
            for (int c = 0; c < NC; ++c) a[c] *= p.scale;
        } else {
            ld_bf16<NC>(p.K + ro, a);
            ld_bf16<NC>(p.V + ro, b);
#pragma unroll
            for (int c = 0; c < NC; ++c) a[c] *= p.scale;
        }
    }
};

// What one edge gathers: Q side k_j, v_j; KV side q_i, dO_i, L_i, Delta_i.
template <int SIDE, int NC>
struct GtEdge {
    Raw<__nv_bfloat16, NC> u;   // Q: k_j; KV: q_i
    Raw<__nv_bfloat16, NC> v;   // Q: v_j
    Raw<float, NC> g;           // KV: dO_i
    float L, Dl;
    __device__ __forceinline__ void load(const GtRunArgs &p, int32_t k, int ch, int hd) {
        const int64_t ko = (int64_t)k * p.HD + ch;
        if constexpr (SIDE == GT_Q) {
            u.load(p.K, ko);
            v.load(p.V, ko);
        } else {
            u.load(p.Q, ko);
            g.load(p.dO, ko);
            L = __ldg(p.lse + (int64_t)k * p.heads + hd);
            Dl = __ldg(p.delta + (int64_t)k * p.heads + hd);
        }
    }
};

// The edges [eb, ee) of one row (gathers one edge ahead of the arithmetic);
// acc holds W = NC (Q: dQ) or 2 NC (KV: dK then dV) floats.
template <int SIDE, int NC, int LPH>
__device__ __forceinline__ void gt_edges(const GtRunArgs &p, const GtRow<SIDE, NC, LPH> &R, int lane, int ch,
                                         int hd, int lph, int32_t eb, int32_t ee, float *acc) {
    if (eb >= ee) return;
    int32_t base = eb;
    int32_t cn = base + lane < ee ? __ldg(p.colidx + base + lane) : 0;
    GtEdge<SIDE, NC> nxt;
    nxt.load(p, __shfl_sync(0xffffffffu, cn, 0), ch, hd);
    for (int32_t e = eb; e < ee; ++e) {
        const GtEdge<SIDE, NC> cur = nxt;
        if (e + 1 < ee) {
            if (e + 1 - base == 32) {
                base = e + 1;
                cn = base + lane < ee ? __ldg(p.colidx + base + lane) : 0;
            }
            nxt.load(p, __shfl_sync(0xffffffffu, cn, e + 1 - base), ch, hd);
        }
        float x[NC], y[NC];
        cur.u.unpack(x);  // Q: k_j; KV: q_i
        if constexpr (SIDE == GT_Q) cur.v.unpack(y);  // v_j
        else cur.g.unpack(y);                         // dO_i
        // s = <q, k> (the scale sits in the row's q or k); da = <dO_i, v_j>
        uint64_t s2 = pk2(0.f, 0.f), d2 = pk2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
            s2 = fma2(pk2(R.a[c], R.a[c + 1]), pk2(x[c], x[c + 1]), s2);
            if constexpr (SIDE == GT_Q) d2 = fma2(pk2(R.b[c], R.b[c + 1]), pk2(y[c], y[c + 1]), d2);
            else d2 = fma2(pk2(y[c], y[c + 1]), pk2(R.b[c], R.b[c + 1]), d2);
        }
        float s0, s1, d0, d1;
        upk2(s2, s0, s1);
        upk2(d2, d0, d1);
        const float sc = head_sum<LPH>(s0 + s1, lph);
        const float da = head_sum<LPH>(d0 + d1, lph);
        if constexpr (SIDE == GT_Q) {
            const float ds = __expf(sc - R.L) * (da - R.Dl);
            const uint64_t ds2 = pk2(ds, ds);
#pragma unroll
            for (int c = 0; c < NC; c += 2)
                upk2(fma2(ds2, pk2(x[c], x[c + 1]), pk2(acc[c], acc[c + 1])), acc[c], acc[c + 1]);
        } else {
            const float al = __expf(sc - cur.L);
            const float ds = al * (da - cur.Dl);
            const uint64_t al2 = pk2(al, al), ds2 = pk2(ds, ds);
#pragma unroll
            for (int c = 0; c < NC; c += 2) {
                upk2(fma2(ds2, pk2(x[c], x[c + 1]), pk2(acc[c], acc[c + 1])), acc[c], acc[c + 1]);
                upk2(fma2(al2, pk2(y[c], y[c + 1]), pk2(acc[NC + c], acc[NC + c + 1])), acc[NC + c],
                     acc[NC + c + 1]);
            }
        }
    }
}

// Store a finished gradient row: Q dQ = scale acc; KV dK = scale acc[0:NC],
// dV = acc[NC:2NC].
template <int SIDE, int NC>
__device__ __forceinline__ void gt_store(const GtRunArgs &p, int32_t r, int ch, const float *acc) {
    const int64_t ro = (int64_t)r * p.HD + ch;
    float t[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) t[c] = acc[c] * p.scale;
    st_f32<NC>(p.dA + ro, t);
    if constexpr (SIDE == GT_KV) st_f32<NC>(p.dB + ro, acc + NC);
}

// A piece of heavy row r leaves its W floats a lane in its slot; the last of
// the row's pieces to arrive sums them in edge order and stores the row.
template <int SIDE, int NC>
__device__ __forceinline__ void gt_flush_piece(const GtRunArgs &p, int64_t w, int32_t r, int lane, int ch,
                                               const float *acc) {
    constexpr int W = SIDE == GT_Q ? NC : 2 * NC;
    const int64_t stride = 2 * (int64_t)p.HD;
    const int32_t rb = __ldg(p.rowptr + r), re = __ldg(p.rowptr + r + 1);
    const int64_t wa = rb / kGatE, wb = ((int64_t)re - 1) / kGatE;
    float *slot = p.slots + (2 * w + (w == wa ? 1 : 0)) * stride + (int64_t)lane * W;
#pragma unroll
    for (int c = 0; c < W; ++c) __stcg(slot + c, acc[c]);
    __threadfence();
    __syncwarp();
    int t = 0;
    if (lane == 0) t = atomicAdd(p.tickets + wa, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t != (int)(wb - wa)) return;
    __threadfence();
    float sum[W];
#pragma unroll
    for (int c = 0; c < W; ++c) sum[c] = 0.f;
    for (int64_t k = wa; k <= wb; ++k) {
        const float *sk = p.slots + (2 * k + (k == wa ? 1 : 0)) * stride + (int64_t)lane * W;
#pragma unroll
        for (int c = 0; c < W; ++c) sum[c] += __ldcg(sk + c);
    }
    gt_store<SIDE, NC>(p, r, ch, sum);
    __syncwarp();
    if (lane == 0) p.tickets[wa] = 0;
}

// resident 256-thread blocks per SM asked of the compiler, per side (the KV
// side holds dK and dV, 16 accumulators a lane at 8 channels: at 3 blocks it
// spills 128 bytes yet runs the R-MAT scale 20 backward in 8.28 ms against
// 9.70 at 2 blocks)
#ifndef GNN_GT_RUN_MINB
#define GNN_GT_RUN_MINB 3
#endif
#ifndef GNN_GT_RUN_MINB_KV
#define GNN_GT_RUN_MINB_KV 3
#endif

template <int SIDE, int NC, int LPH>
__global__ void __launch_bounds__(kGatWarps * 32, SIDE == GT_Q ? GNN_GT_RUN_MINB : GNN_GT_RUN_MINB_KV)
k_gt_bwd_run(GtRunArgs p) {
    constexpr int W = SIDE == GT_Q ? NC : 2 * NC;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t w = (int64_t)blockIdx.x * kGatWarps + warp;
    if (w >= p.n_runs) return;
    const int lph = LPH > 0 ? LPH : p.D / NC;
    const int ch = lane * NC;
    const int hd = ch / p.D;
    const int64_t e0 = w * kGatE, e1 = min(e0 + kGatE, p.nnz);
    const int32_t lo = __ldg(p.run_rows + w), lo_end = __ldg(p.run_rows + w + 1);
    // a heavy row that started in an earlier run and reaches into this one
    if (lo > 0 && e0 < p.nnz) {
        const int32_t lo_beg = __ldg(p.rowptr + lo);
        if (lo_beg > e0 && lo_beg - __ldg(p.rowptr + lo - 1) > kGatE) {
            GtRow<SIDE, NC, LPH> R;
            R.load(p, lo - 1, ch, hd, lph, true);
            float acc[W];
#pragma unroll
            for (int c = 0; c < W; ++c) acc[c] = 0.f;
            gt_edges<SIDE, NC, LPH>(p, R, lane, ch, hd, lph, (int32_t)e0, (int32_t)min((int64_t)lo_beg, e1), acc);
            gt_flush_piece<SIDE, NC>(p, w, lo - 1, lane, ch, acc);
        }
    }
    // owned rows, bounds read 32 at a time
    for (int32_t rbase = lo; rbase < lo_end; rbase += 32) {
        const int32_t rr = rbase + lane;
        int32_t my_b = 0, my_e = 0;
        if (rr < lo_end) {
            my_b = __ldg(p.rowptr + rr);
            my_e = __ldg(p.rowptr + rr + 1);
        }
        const int cnt = min(32, lo_end - rbase);
        for (int k = 0; k < cnt; ++k) {
            const int32_t r = rbase + k;
            const int32_t rb = __shfl_sync(0xffffffffu, my_b, k), re = __shfl_sync(0xffffffffu, my_e, k);
            GtRow<SIDE, NC, LPH> R;
            R.load(p, r, ch, hd, lph, re > rb);
            if constexpr (SIDE == GT_Q) {
                if (lane % lph == 0) p.delta[(int64_t)r * p.heads + hd] = R.Dl;
            }
            float acc[W];
#pragma unroll
            for (int c = 0; c < W; ++c) acc[c] = 0.f;
            if (re - rb > kGatE) {  // heavy: its first piece (the last owned row)
                gt_edges<SIDE, NC, LPH>(p, R, lane, ch, hd, lph, rb, (int32_t)e1, acc);
                gt_flush_piece<SIDE, NC>(p, w, r, lane, ch, acc);
            } else {
                gt_edges<SIDE, NC, LPH>(p, R, lane, ch, hd, lph, rb, re, acc);
                gt_store<SIDE, NC>(p, r, ch, acc);
            }
        }
    }
}

struct GatBwdWs {
    float *G, *slots, *da_part, *da_part2;
    int32_t *run_rows, *run_rows_t, *tickets, *da_ticket;
    size_t bytes;
};

// Channels per lane: a warp covers 32 NC channels, one channel group (grid
// y).  Rows of up to 256 channels are one group: splitting a 256-channel row
// over two warps of 4 channels a lane was slower on R-MAT scale 20 (4 heads
// x 64: 11.6 ms at the best occupancy against 9.3 ms), since every edge then
// costs each warp its index, score reductions and exponential again.
constexpr int kGatMaxNC = 8;
inline int gat_nc(int32_t HD) { return std::min(HD / 32, kGatMaxNC); }
inline int gat_groups(int32_t HD) { return HD / (32 * gat_nc(HD)); }

GatBwdWs gat_bwd_layout(const gnn_csr *g, int32_t heads, int32_t HD, void *base) {
    const int64_t nr = n_runs(g->nnz, (int32_t)kGatE);
    const int64_t blocks = (nr + kGatWarps - 1) / kGatWarps;
    GatBwdWs W{};
    char *b = static_cast<char *>(base);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        char *q = b ? b + o : nullptr;
        o = round_up(o + bytes, 256);
        return q;
    };
    W.G = reinterpret_cast<float *>(take(sizeof(float) * (size_t)std::max<int64_t>((int64_t)g->n_rows * heads, 1)));
    W.slots = reinterpret_cast<float *>(take(sizeof(float) * (size_t)(2 * nr) * HD));
    W.da_part = reinterpret_cast<float *>(take(sizeof(float) * (size_t)blocks * HD));
    W.da_part2 = reinterpret_cast<float *>(take(sizeof(float) * (size_t)kDaBlocks * HD));
    W.run_rows = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)(nr + 1)));
    W.run_rows_t = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)(nr + 1)));
    W.tickets = reinterpret_cast<int32_t *>(take(sizeof(int32_t) * (size_t)nr * gat_groups(HD)));
    W.da_ticket = reinterpret_cast<int32_t *>(take(sizeof(int32_t)));
    W.bytes = o;
    return W;
}

template <typename T, int NC>
void launch_gatv2_bwd(const GatBwdArgs &al, const GatBwdArgs &r, const GatBwdWs &W, float *da, cudaStream_t s) {
    const int blocks = (int)((al.n_runs + kGatWarps - 1) / kGatWarps);
    const dim3 grid(blocks, gat_groups(al.HD));
    const int64_t nt = (int64_t)al.n + 1;
    k_gatv2_bwd_runs<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(al.rowptr, r.rowptr, al.n, al.n_runs, W.run_rows,
                                                                   W.run_rows_t, W.tickets,
                                                                   al.n_runs * gat_groups(al.HD), W.da_ticket);
    // lanes per head fixed at compile time for the 8-channel shapes (4 or 8
    // lanes: 32- or 64-dimensional heads), a runtime value otherwise
    const int lph = al.D / NC;
    if (NC == 8 && lph == 8) {
        k_gatv2_bwd<GAT_AL, T, NC, 8><<<grid, kGatWarps * 32, 0, s>>>(al);
        k_gatv2_bwd<GAT_R, T, NC, 8><<<grid, kGatWarps * 32, 0, s>>>(r);
    } else if (NC == 8 && lph == 4) {
        k_gatv2_bwd<GAT_AL, T, NC, 4><<<grid, kGatWarps * 32, 0, s>>>(al);
        k_gatv2_bwd<GAT_R, T, NC, 4><<<grid, kGatWarps * 32, 0, s>>>(r);
    } else {
        k_gatv2_bwd<GAT_AL, T, NC, 0><<<grid, kGatWarps * 32, 0, s>>>(al);
        k_gatv2_bwd<GAT_R, T, NC, 0><<<grid, kGatWarps * 32, 0, s>>>(r);
    }
    k_gatv2_bwd_da<<<kDaBlocks, 256, 0, s>>>(W.da_part, blocks, al.HD, W.da_part2, W.da_ticket, da);
}

// Schedule of the GT backward: 1 = a warp per row, 2 = edge runs, 0 = by
// the graph's mean degree (runs below GNN_GT_RUNS_BELOW_DEGREE: power-law
// graphs, whose hub rows would leave one warp with tens of thousands of
// edges; a warp per row where rows are long and even).  Measured on GB300
// (8 heads x 32, bf16): R-MAT scale 20 (mean degree 16, max 39,472) 43.0 ms
// per row against 8.3 ms on runs; the clustered 262K-node graph (mean 77)
// 4.04 ms per row against 4.96 ms on runs.
#ifndef GNN_GT_BWD_SCHEDULE
#define GNN_GT_BWD_SCHEDULE 0
#endif
#ifndef GNN_GT_RUNS_BELOW_DEGREE
#define GNN_GT_RUNS_BELOW_DEGREE 32
#endif
inline bool gt_bwd_use_runs(const gnn_csr *g) {
    if (GNN_GT_BWD_SCHEDULE == 1) return false;
    if (GNN_GT_BWD_SCHEDULE == 2) return true;
    return g->nnz < (int64_t)GNN_GT_RUNS_BELOW_DEGREE * g->n_rows;
}

struct GtBwdWs {
    float *delta, *slots;
    int32_t *run_rows, *run_rows_t, *tickets, *spare;
    size_t bytes;
};

GtBwdWs gt_bwd_layout(const gnn_csr *g, int32_t heads, int32_t HD, void *base) {
    const int64_t nr = n_runs(g->nnz, (int32_t)kGatE);
    Carver cv(base);
    GtBwdWs W{};
    W.delta = cv.take<float>((size_t)std::max<int64_t>((int64_t)g->n_rows * heads, 1));
    W.slots = cv.take<float>((size_t)(2 * nr) * 2 * HD);
    W.run_rows = cv.take<int32_t>((size_t)(nr + 1));
    W.run_rows_t = cv.take<int32_t>((size_t)(nr + 1));
    W.tickets = cv.take<int32_t>((size_t)nr);
    W.spare = cv.take<int32_t>(1);
    W.bytes = cv.used;
    return W;
}

// Warp per row: dQ and Delta over the CSR, then dK and dV over CSR^T.
template <int NC>
void launch_gt_bwd_rows(const GtBwdArgs &q, const GtBwdArgs &kv, cudaStream_t s) {
    const int blocks = (int)(((int64_t)q.n * 32 + 255) / 256);
    const int lph = q.D / NC;
    if (NC == 8 && lph == 4) {
        k_gt_bwd_q<NC, 4><<<blocks, 256, 0, s>>>(q);
        k_gt_bwd_kv<NC, 4><<<blocks, 256, 0, s>>>(kv);
    } else if (NC == 8 && lph == 8) {
        k_gt_bwd_q<NC, 8><<<blocks, 256, 0, s>>>(q);
        k_gt_bwd_kv<NC, 8><<<blocks, 256, 0, s>>>(kv);
    } else {
        k_gt_bwd_q<NC, 0><<<blocks, 256, 0, s>>>(q);
        k_gt_bwd_kv<NC, 0><<<blocks, 256, 0, s>>>(kv);
    }
}

// Edge runs: run tables of CSR and CSR^T (and the tickets cleared), then dQ
// and Delta over the CSR, then dK and dV over CSR^T
template <int NC, int LPH>
void launch_gt_bwd(const GtRunArgs &q, const GtRunArgs &kv, const GtBwdWs &W, cudaStream_t s) {
    const int64_t nt = (int64_t)q.n + 1;
    k_gatv2_bwd_runs<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(q.rowptr, kv.rowptr, q.n, q.n_runs, W.run_rows,
                                                                   W.run_rows_t, W.tickets, q.n_runs, W.spare);
    const int blocks = (int)((q.n_runs + kGatWarps - 1) / kGatWarps);
    k_gt_bwd_run<GT_Q, NC, LPH><<<blocks, kGatWarps * 32, 0, s>>>(q);
    k_gt_bwd_run<GT_KV, NC, LPH><<<blocks, kGatWarps * 32, 0, s>>>(kv);
}

}  // namespace

size_t gt_bwd_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim) {
    if (heads <= 0 || head_dim <= 0) return 0;
    return gt_bwd_layout(g, heads, heads * head_dim, nullptr).bytes;
}

size_t gatv2_bwd_workspace_bytes(const gnn_csr *g, int32_t heads, int32_t head_dim) {
    if (heads <= 0 || head_dim <= 0) return 0;
    return gat_bwd_layout(g, heads, heads * head_dim, nullptr).bytes;
}

}  // namespace gnn

using namespace gnn;

extern "C" gnn_status gnn_gt_attn_bwd(const gnn_csr *g, const gnn_csr *gt, const void *Q, const void *K,
                                      const void *V, int32_t dtype, int32_t heads, int32_t head_dim, float scale,
                                      const float *out, const float *lse, const float *dout, float *dQ,
                                      float *dK, float *dV, void *ws, size_t ws_bytes, void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    st = check_csr_args(gt);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols || gt->n_rows != g->n_cols || gt->n_cols != g->n_rows || gt->nnz != g->nnz)
        return GNN_ERR_INVALID_ARG;
    if (dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    if (heads <= 0 || head_dim <= 0) return GNN_ERR_INVALID_ARG;
    const int32_t HD = heads * head_dim;
    if (HD != 128 && HD != 256) return GNN_ERR_UNSUPPORTED;
    const int NC = HD / 32;
    const int lph = head_dim / NC;
    if (head_dim % NC || lph < 1 || (lph & (lph - 1))) return GNN_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !out || !lse || !dout || !dQ || !dK || !dV) return GNN_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
        return GNN_ERR_INVALID_ARG;
    if (!ws || ws_bytes < gt_bwd_workspace_bytes(g, heads, head_dim)) return GNN_ERR_WORKSPACE;
    if (g->n_rows == 0) return GNN_OK;

    const GtBwdWs W = gt_bwd_layout(g, heads, HD, ws);
    GtRunArgs q{};
    q.rowptr = g->rowptr;
    q.colidx = g->colidx;
    q.run_rows = W.run_rows;
    q.Q = static_cast<const __nv_bfloat16 *>(Q);
    q.K = static_cast<const __nv_bfloat16 *>(K);
    q.V = static_cast<const __nv_bfloat16 *>(V);
    q.O = out;
    q.lse = lse;
    q.dO = dout;
    q.delta = W.delta;
    q.dA = dQ;
    q.slots = W.slots;
    q.tickets = W.tickets;
    q.nnz = g->nnz;
    q.n_runs = n_runs(g->nnz, (int32_t)kGatE);
    q.n = g->n_rows;
    q.heads = heads;
    q.D = head_dim;
    q.HD = HD;
    q.scale = scale;
    GtRunArgs kv = q;
    kv.rowptr = gt->rowptr;
    kv.colidx = gt->colidx;
    kv.run_rows = W.run_rows_t;
    kv.dA = dK;
    kv.dB = dV;
    cudaStream_t s = as_stream(stream);
    if (!gt_bwd_use_runs(g)) {
        GtBwdArgs qr{};
        qr.rowptr = g->rowptr;
        qr.colidx = g->colidx;
        qr.Q = q.Q;
        qr.K = q.K;
        qr.V = q.V;
        qr.O = out;
        qr.lse = lse;
        qr.dO = dout;
        qr.delta = W.delta;
        qr.dA = dQ;
        qr.n = g->n_rows;
        qr.heads = heads;
        qr.D = head_dim;
        qr.HD = HD;
        qr.scale = scale;
        GtBwdArgs kvr = qr;
        kvr.rowptr = gt->rowptr;
        kvr.colidx = gt->colidx;
        kvr.dA = dK;
        kvr.dB = dV;
        if (NC == 4) launch_gt_bwd_rows<4>(qr, kvr, s);
        else launch_gt_bwd_rows<8>(qr, kvr, s);
        note_launch(2);
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }
    if (NC == 8 && lph == 4) launch_gt_bwd<8, 4>(q, kv, W, s);
    else if (NC == 8 && lph == 8) launch_gt_bwd<8, 8>(q, kv, W, s);
    else if (NC == 8) launch_gt_bwd<8, 0>(q, kv, W, s);
    else launch_gt_bwd<4, 0>(q, kv, W, s);
    note_launch(3);
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}

extern "C" gnn_status gnn_gatv2_attn_bwd(const gnn_csr *g, const gnn_csr *gt, const void *Cl, const void *Cr,
                                        int32_t dtype, const float *a, int32_t heads, int32_t head_dim,
                                        float neg_slope, const float *out, const float *lse, const float *dout,
                                        float *dl, float *dr, float *da, void *ws, size_t ws_bytes,
                                        void *stream) {
    gnn_status st = check_csr_args(g);
    if (st != GNN_OK) return st;
    st = check_csr_args(gt);
    if (st != GNN_OK) return st;
    if (g->n_rows != g->n_cols || gt->n_rows != g->n_cols || gt->n_cols != g->n_rows || gt->nnz != g->nnz)
        return GNN_ERR_INVALID_ARG;
    if (dtype != GNN_F32 && dtype != GNN_BF16) return GNN_ERR_UNSUPPORTED;
    if (heads <= 0 || head_dim <= 0) return GNN_ERR_INVALID_ARG;
    const int32_t HD = heads * head_dim;
    if (HD != 32 && HD != 64 && HD != 128 && HD != 256) return GNN_ERR_UNSUPPORTED;
    const int NC = gat_nc(HD);
    const int lph = head_dim / NC;
    // a head lies within one warp's channel group, on a power of two of lanes
    if (head_dim % NC || (32 * NC) % head_dim || (lph & (lph - 1))) return GNN_ERR_UNSUPPORTED;
    if (!Cl || !Cr || !a || !out || !lse || !dout || !dl || !dr || !da) return GNN_ERR_INVALID_ARG;
    if (!aligned16(Cl) || !aligned16(Cr) || !aligned16(a) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dl) || !aligned16(dr))
        return GNN_ERR_INVALID_ARG;
    if (!ws || ws_bytes < gatv2_bwd_workspace_bytes(g, heads, head_dim)) return GNN_ERR_WORKSPACE;
    if (g->n_rows == 0) {
        cudaStream_t s = as_stream(stream);
        if (cudaMemsetAsync(da, 0, sizeof(float) * (size_t)HD, s) != cudaSuccess) return GNN_ERR_CUDA;
        return GNN_OK;
    }
    const GatBwdWs W = gat_bwd_layout(g, heads, HD, ws);
    GatBwdArgs al{};
    al.rowptr = g->rowptr;
    al.colidx = g->colidx;
    al.run_rows = W.run_rows;
    al.Cl = Cl;
    al.Cr = Cr;
    al.a = a;
    al.O = out;
    al.lse = lse;
    al.dO = dout;
    al.G = W.G;
    al.grad = dl;
    al.slots = W.slots;
    al.tickets = W.tickets;
    al.da_part = W.da_part;
    al.nnz = g->nnz;
    al.n_runs = n_runs(g->nnz, (int32_t)kGatE);
    al.n = g->n_rows;
    al.heads = heads;
    al.D = head_dim;
    al.HD = HD;
    al.slope = neg_slope;
    GatBwdArgs r = al;
    r.rowptr = gt->rowptr;
    r.colidx = gt->colidx;
    r.run_rows = W.run_rows_t;
    r.grad = dr;
    r.da_part = nullptr;
    cudaStream_t s = as_stream(stream);
    const bool bf = dtype == GNN_BF16;
    switch (NC) {
        case 1: bf ? launch_gatv2_bwd<__nv_bfloat16, 1>(al, r, W, da, s) : launch_gatv2_bwd<float, 1>(al, r, W, da, s); break;
        case 2: bf ? launch_gatv2_bwd<__nv_bfloat16, 2>(al, r, W, da, s) : launch_gatv2_bwd<float, 2>(al, r, W, da, s); break;
        case 4: bf ? launch_gatv2_bwd<__nv_bfloat16, 4>(al, r, W, da, s) : launch_gatv2_bwd<float, 4>(al, r, W, da, s); break;
        default: bf ? launch_gatv2_bwd<__nv_bfloat16, 8>(al, r, W, da, s) : launch_gatv2_bwd<float, 8>(al, r, W, da, s); break;
    }
    note_launch(4);
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}
