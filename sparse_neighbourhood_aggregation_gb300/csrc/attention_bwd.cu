// Backward of the fused Graph Transformer attention.
//
// IO-aware GNN layers, Appendix D.2 (the GT backward: Delta = <O, dO> per
// destination and head in a kernel of its own, then the kernels over CSR and
// CSR^T that recompute the weights from the stored logsumexp L).  For row i,
// head h, edge j in N(i), with s_ij = scale <q_i, k_j>:
//   alpha_ij = exp(s_ij - L_i),  ds_ij = alpha_ij (<dO_i, v_j> - Delta_i)
//   dQ_i = scale sum_j ds_ij k_j          (k_gt_bwd_q, a warp per row of CSR)
//   dK_j = scale sum_i ds_ij q_i,  dV_j = sum_i alpha_ij dO_i
//                                        (k_gt_bwd_kv, a warp per row of CSR^T)
// Each gradient row is owned by one warp, so there are no atomics and the
// sums are deterministic.  Lane l holds channels [l*NC, (l+1)*NC) of the
// HD = 32 NC channels; the D / NC lanes of a head reduce its dot products
// with shuffles.  The edge loop loads the rows of U edges before using any.
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
constexpr int kBwdU = 1;

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

// sum over the lph lanes of this lane's head (lph a power of two)
__device__ __forceinline__ float head_sum(float x, int lph) {
    for (int o = lph >> 1; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <int NC>
__global__ void __launch_bounds__(256) k_gt_bwd_q(GtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int32_t i = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (i >= a.n) return;
    const int lph = a.D / NC;
    const int h = (lane * NC) / a.D;
    const int64_t ro = (int64_t)i * a.HD + lane * NC;
    float q[NC], o[NC], g[NC], dq[NC];
    ld_bf16<NC>(a.Q + ro, q);
    ld_f32<NC>(a.O + ro, o);
    ld_f32<NC>(a.dO + ro, g);
    float p = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        p = fmaf(o[c], g[c], p);
        q[c] *= a.scale;
        dq[c] = 0.f;
    }
    const float delta = head_sum(p, lph);
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
                float s = 0.f, da = 0.f;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    s = fmaf(q[c], kf[u][c], s);
                    da = fmaf(g[c], vf[u][c], da);
                }
                s = head_sum(s, lph);
                da = head_sum(da, lph);
                const float ds = __expf(s - L) * (da - delta);
#pragma unroll
                for (int c = 0; c < NC; ++c) dq[c] = fmaf(ds, kf[u][c], dq[c]);
            }
        }
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) dq[c] *= a.scale;
    st_f32<NC>(a.dA + ro, dq);
    if (lane % lph == 0) a.delta[(int64_t)i * a.heads + h] = delta;
}

template <int NC>
__global__ void __launch_bounds__(256) k_gt_bwd_kv(GtBwdArgs a) {
    const int lane = threadIdx.x & 31;
    const int32_t j = (int32_t)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    if (j >= a.n) return;
    const int lph = a.D / NC;
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
                float s = 0.f, da = 0.f;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    s = fmaf(qf[u][c], kf[c], s);
                    da = fmaf(gf[u][c], vf[c], da);
                }
                s = head_sum(s, lph);
                da = head_sum(da, lph);
                const float al = __expf(s - Lh[u]);
                const float ds = al * (da - Dh[u]);
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    dv[c] = fmaf(al, gf[u][c], dv[c]);
                    dk[c] = fmaf(ds, qf[u][c], dk[c]);
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

template <int NC>
void launch_gt_bwd(GtBwdArgs q, GtBwdArgs kv, cudaStream_t s) {
    const int blocks = (int)(((int64_t)q.n * 32 + 255) / 256);
    k_gt_bwd_q<NC><<<blocks, 256, 0, s>>>(q);
    k_gt_bwd_kv<NC><<<blocks, 256, 0, s>>>(kv);
}

}  // namespace

size_t gt_bwd_workspace_bytes(const gnn_csr *g, int32_t heads) {
    return round_up(sizeof(float) * (size_t)std::max<int64_t>((int64_t)g->n_rows * heads, 1), 256);
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
    if (!ws || ws_bytes < gt_bwd_workspace_bytes(g, heads)) return GNN_ERR_WORKSPACE;
    if (g->n_rows == 0) return GNN_OK;

    GtBwdArgs q{};
    q.rowptr = g->rowptr;
    q.colidx = g->colidx;
    q.Q = static_cast<const __nv_bfloat16 *>(Q);
    q.K = static_cast<const __nv_bfloat16 *>(K);
    q.V = static_cast<const __nv_bfloat16 *>(V);
    q.O = out;
    q.lse = lse;
    q.dO = dout;
    q.delta = static_cast<float *>(ws);
    q.dA = dQ;
    q.n = g->n_rows;
    q.heads = heads;
    q.D = head_dim;
    q.HD = HD;
    q.scale = scale;
    GtBwdArgs kv = q;
    kv.rowptr = gt->rowptr;
    kv.colidx = gt->colidx;
    kv.dA = dK;
    kv.dB = dV;
    cudaStream_t s = as_stream(stream);
    if (NC == 4) launch_gt_bwd<4>(q, kv, s);
    else launch_gt_bwd<8>(q, kv, s);
    note_launch(2);
    GNN_LAUNCH_CHECK();
    return GNN_OK;
}
