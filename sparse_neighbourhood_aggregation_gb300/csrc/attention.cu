// Steps a4 (fused GATv2 forward) and a5 (fused Graph Transformer attention,
// CSR path), plus the SIMT projection used where the tensor-core path does
// not apply.
//
// IO-aware GNN layers, Section 2.2 (iii) (GATv2 and GT scores), Section 3.2
// and Appendix D.2 (fused CSR forward: score, online softmax and weighted
// aggregate in one pass over the destination's adjacency list, logsumexp kept
// for the backward pass; no per-edge score, weight or message reaches HBM).
//
// GB300 design.
// * Schedule: one warp is one worker.  The edge list is cut into runs of E
//   edges (the prepared graph's run table, read at a stride); a warp owns the
//   rows whose first edge lies in its run and processes each of them whole,
//   so short rows of a power-law graph are packed many to a warp.  A row
//   longer than E (heavy) is cut at run boundaries; every piece leaves its
//   softmax state (running max, running sum, unnormalised accumulator) in a
//   workspace slot, and the last piece to finish (ticket counter, no
//   spinning) merges the pieces in edge order, so the result does not depend
//   on scheduling.  A run can hold the last piece of one heavy row and the
//   first piece of the next, so each run has two slots: 2w for a piece
//   continued from an earlier run, 2w+1 for the first piece of a row it owns.
// * Gathers: the warp's edges (one contiguous span) stream through a ring of
//   S shared-memory stages of U neighbour records.  Lane u of the warp
//   fetches the record of edge u of a batch with one bulk copy
//   (cp.async.bulk, completing on the stage's mbarrier), S batches ahead of
//   their use, with the column ids of the next batch prefetched.  The data in
//   flight sits in shared memory, not registers, and the TMA engine does the
//   address work.  A GATv2 record is the projected row r_j followed by its
//   per-head linear parts A_r[j] (one copy); a GT record is K_j then V_j.
//   (Filling the ring with 16-byte cp.async copies instead, 32/U lanes per
//   record, issues ~8 fewer instructions per edge but measured 5-15% slower
//   on GB300.)
// * Softmax: the running maximum moves only when a score exceeds it by more
//   than kLazy (base-2 units), so the rescale of the accumulator (a multiply
//   per channel and an exp2) is rare; weights stay below 2^kLazy.
// * Lanes: lane l owns CPL consecutive 16-byte chunks of a feature row (8
//   bf16 or 4 fp32 channels per chunk); a head's channels sit on
//   D / (CPL * chunk) adjacent lanes, whose partial scores are summed with
//   xor-shuffles.  Scores are kept in base-2 units (scaled by log2 e) so each
//   softmax weight is a single exp2.  Edges are scored four at a time where a
//   row allows, so the shuffle chains of four edges overlap.
//
// GATv2 score.  With LeakyReLU slope s, LReLU(x) = (1+s)/2 x + (1-s)/2 |x|,
// so  e_ij = A_l[i] + A_r[j] + sum_d a''_d |l_id + r_jd|  with
// A_l[i,h] = sum_d a'_hd l_id, A_r[j,h] = sum_d a'_hd r_jd, a' = (1+s)/2 a,
// a'' = (1-s)/2 a.  A_l and A_r are per-node scalars formed once with the
// projection; per edge and channel only an add and an |.| multiply-add remain
// (the plain definition needs add, multiply, max and multiply-add).
#include <algorithm>
#include <mutex>

#include "async.cuh"
#include "common.cuh"

namespace gnn {

gnn_status check_csr_args(const gnn_csr *g);
const int32_t *prep_run_table(const gnn_csr *g, const void *prep);

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// lazy-rescale margin of the online softmax (base-2 units); measured on
// GB300 against a rescale at every new maximum: GATv2 attention at R-MAT
// scale 20 2.064 -> 2.054 ms, GT on the clustered graph 2.107 -> 2.080 ms
constexpr float kLazy = 8.f;
// attention run = kAttnRunMul runs of the prepared graph's run table
constexpr int kAttnRunMul = 4;
constexpr int kAttnE = kRunEdges * kAttnRunMul;
constexpr int kAttnWarps = 4;  // warps per block
// Edges scored together and resident 4-warp blocks per SM asked of the
// compiler, per attention kind (measured on GB300: GATv2 at c3, 2 edges and
// 6 blocks, 2.07 ms against 2.32 ms for 4 edges at the compiler's choice of
// 127 registers; GT at c4, 4 edges and 5 blocks, 2.11 against 2.32 ms).
// Lanes holding more than 8 channels (wide fp32 heads) keep 4-edge groups
// and the compiler's register choice.
__host__ __device__ constexpr int att_group(int kind, int nc) { return (kind == 0 && nc <= 8) ? 2 : 4; }
__host__ __device__ constexpr int att_min_blocks(int kind, int nc) { return nc > 8 ? 1 : kind == 0 ? 6 : 5; }

enum AttnKind { ATT_GATV2 = 0, ATT_GT = 1 };

// floats per softmax-state slot: HD accumulator channels then (m, s) per
// head, rounded up to 16 bytes so every slot starts 16-byte aligned
__host__ __device__ __forceinline__ int64_t slot_stride(int32_t HD, int32_t heads) {
    return ((int64_t)HD + 2 * heads + 3) & ~(int64_t)3;
}

// bytes of a projected GATv2 row: HD channels then A[heads] fp32, padded
// to 16 bytes (rows are bulk-copied whole)
__host__ __device__ __forceinline__ int64_t gat_row_bytes(int32_t HD, int32_t heads, int32_t esize) {
    return (int64_t)HD * esize + (((int64_t)heads * 4 + 15) & ~(int64_t)15);
}

struct AttnArgs {
    const int32_t *rowptr;
    const int32_t *colidx;
    const int32_t *run_table;  // prepared graph's run table (E = kRunEdges) or null
    const char *Sg;            // gathered rows: GATv2 padded r rows, GT K
    const char *Vg;            // GT V (GATv2 unused)
    const char *Qd;            // destination rows: GATv2 padded l rows, GT Q
    int64_t sg_stride, vg_stride, qd_stride;  // bytes between rows
    int32_t s_bytes, v_bytes;  // bytes copied per edge from Sg and Vg
    int32_t rec;               // bytes of one edge record in the ring
    int32_t ar_off;            // GATv2: offset of A within a padded row
    int32_t U, S;              // edges per stage, stages
    int32_t ring_bytes;        // per warp: S*U*rec + S mbarriers
    const float *coef;         // GATv2 [HD] (1-s)/2 a log2e
    float qscale;              // GT: scale * log2e
    float *out;                // [n_rows, HD]
    float *lse;                // [n_rows, heads] or null
    float *slots;              // [2 n_workers, slot_stride]
    int32_t *tickets;          // [n_workers], zero on entry and on exit
    int32_t *err;              // device error word
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

template <int KIND, class T, int CPL, int LPH>
struct Lane {
    static constexpr int NV = Elt<T>::N;
    static constexpr int NC = CPL * NV;  // channels per lane
    int lane;
    bool active;  // owns channels
    int head;     // head of the lane's channels
    int lph;      // lanes per head (when LPH == 0)
    float coef[KIND == ATT_GATV2 ? NC : 1];
    // lanes per head: the template constant, or the runtime value if 0
    __device__ __forceinline__ int lphv() const { return LPH > 0 ? LPH : lph; }
    // a compile-time LPH is used only when every lane owns channels
    __device__ __forceinline__ bool act() const { return LPH > 0 ? true : active; }
};

// Ring geometry (bytes of an edge record, edges per stage, stages), fixed
// at compile time for GATv2 on bf16 rows of 32 16-byte chunks with a
// compile-time lanes-per-head, where it follows from the template (so the
// per-edge address arithmetic folds); the runtime values of AttnArgs
// otherwise.  Measured on GB300: GATv2 at R-MAT scale 20 2.285 -> 2.147 ms
// for the layer; GT on the clustered graph went 2.08 -> 2.24 ms with it, so
// GT keeps the runtime geometry.
template <int KIND, class T, int CPL, int LPH>
struct Geo {
    static constexpr bool FIXED = KIND == ATT_GATV2 && LPH > 0 && sizeof(T) == 2 && CPL == 1;
    static constexpr int SB = KIND == ATT_GATV2 ? 512 + ((FIXED ? 32 / LPH : 1) * 4 + 15) / 16 * 16 : 512;
    static constexpr int VB = KIND == ATT_GATV2 ? 0 : 512;
    static constexpr int REC = SB + VB;
    static constexpr int UU = REC <= 640 ? 8 : 4;
    static constexpr int SS = 2;
    __host__ __device__ __forceinline__ static int rec(const AttnArgs &a) { return FIXED ? REC : a.rec; }
    __host__ __device__ __forceinline__ static int U(const AttnArgs &a) { return FIXED ? UU : a.U; }
    __host__ __device__ __forceinline__ static int S(const AttnArgs &a) { return FIXED ? SS : a.S; }
    __host__ __device__ __forceinline__ static int s_bytes(const AttnArgs &a) { return FIXED ? SB : a.s_bytes; }
    __host__ __device__ __forceinline__ static int v_bytes(const AttnArgs &a) { return FIXED ? VB : a.v_bytes; }
    __host__ __device__ __forceinline__ static int ar_off(const AttnArgs &a) { return FIXED ? 512 : a.ar_off; }
    // the runtime geometry the host set up agrees with the fixed one
    static bool agrees(const AttnArgs &a) {
        return !FIXED || (a.rec == REC && a.U == UU && a.S == SS && a.s_bytes == SB && a.v_bytes == VB &&
                          (KIND != ATT_GATV2 || a.ar_off == 512));
    }
};

template <class T, int CPL>
__device__ __forceinline__ void unpack_row(const uint4 *v, float *f) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) Chunk<T>::unpack(v[c], f + c * Elt<T>::N);
}

// Score NG edges held in ring records rec0[0..NG) and fold them into st.
// dq: the destination's channels (l for GATv2, Q pre-scaled for GT);
// al: A_l[row, head] (GATv2).
template <int KIND, class T, int CPL, int LPH, int NG>
__device__ __forceinline__ void fold_edges(const AttnArgs &a, const Lane<KIND, T, CPL, LPH> &L,
                                           const unsigned char *rec0, const float *dq, float al,
                                           SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    float sf[NG][NC];
    float part[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const unsigned char *rec = rec0 + g * Geo<KIND, T, CPL, LPH>::rec(a);
        uint4 sv[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            sv[c] = L.act() ? *reinterpret_cast<const uint4 *>(rec + (L.lane * CPL + c) * 16)
                             : make_uint4(0u, 0u, 0u, 0u);
        unpack_row<T, CPL>(sv, sf[g]);
        float p0 = 0.f, p1 = 0.f;  // two chains: half the dependent-FMA latency
        if (KIND == ATT_GATV2) {
#pragma unroll
            for (int k = 0; k < NC; k += 2) {
                float x0, x1;
                upk2(add2(pk2(dq[k], dq[k + 1]), pk2(sf[g][k], sf[g][k + 1])), x0, x1);
                p0 = fmaf(L.coef[k], fabsf(x0), p0);
                p1 = fmaf(L.coef[k + 1], fabsf(x1), p1);
            }
        } else {
            uint64_t pp = pk2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < NC; k += 2) pp = fma2(pk2(dq[k], dq[k + 1]), pk2(sf[g][k], sf[g][k + 1]), pp);
            upk2(pp, p0, p1);
        }
        part[g] = p0 + p1;
    }
    for (int o = L.lphv() >> 1; o > 0; o >>= 1) {
#pragma unroll
        for (int g = 0; g < NG; ++g) part[g] += __shfl_xor_sync(0xffffffffu, part[g], o);
    }
    float mx = st.m;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (KIND == ATT_GATV2)
            part[g] += al + (L.act() ? *reinterpret_cast<const float *>(rec0 + g * Geo<KIND, T, CPL, LPH>::rec(a) +
                                                                         Geo<KIND, T, CPL, LPH>::ar_off(a) + 4 * L.head)
                                      : 0.f);
        mx = fmaxf(mx, part[g]);
    }
    // lazy rescale: a new maximum is taken only kLazy above the current one
    // (-inf + kLazy is -inf, so a head's first score always sets it)
    if (__any_sync(0xffffffffu, mx > st.m + kLazy)) {
        const bool up = mx > st.m + kLazy;
        const float sc = up ? exp2_approx(st.m - mx) : 1.f;
        st.s *= sc;
#pragma unroll
        for (int k = 0; k < NC; ++k) st.acc[k] *= sc;
        if (up) st.m = mx;
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const float p = exp2_approx(part[g] - st.m);
        st.s += p;
        const uint64_t pp = pk2(p, p);
        if (KIND == ATT_GATV2) {
#pragma unroll
            for (int k = 0; k < NC; k += 2)
                upk2(fma2(pp, pk2(sf[g][k], sf[g][k + 1]), pk2(st.acc[k], st.acc[k + 1])), st.acc[k], st.acc[k + 1]);
        } else {
            const unsigned char *rec = rec0 + g * Geo<KIND, T, CPL, LPH>::rec(a) + Geo<KIND, T, CPL, LPH>::s_bytes(a);
            uint4 vv[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                vv[c] = L.act() ? *reinterpret_cast<const uint4 *>(rec + (L.lane * CPL + c) * 16)
                                 : make_uint4(0u, 0u, 0u, 0u);
            float vf[NC];
            unpack_row<T, CPL>(vv, vf);
#pragma unroll
            for (int k = 0; k < NC; k += 2)
                upk2(fma2(pp, pk2(vf[k], vf[k + 1]), pk2(st.acc[k], st.acc[k + 1])), st.acc[k], st.acc[k + 1]);
        }
    }
}

template <int KIND, class T, int CPL, int LPH>
__device__ __forceinline__ void store_final(const AttnArgs &a, const Lane<KIND, T, CPL, LPH> &L, int32_t r,
                                            const SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    if (!L.act()) return;
    const float inv = st.s > 0.f ? 1.f / st.s : 0.f;
    float *o = a.out + (int64_t)r * a.HD + (int64_t)L.lane * NC;
#pragma unroll
    for (int k = 0; k < NC; k += 4)
        *reinterpret_cast<float4 *>(o + k) =
            make_float4(st.acc[k] * inv, st.acc[k + 1] * inv, st.acc[k + 2] * inv, st.acc[k + 3] * inv);
    if (a.lse && (L.lane % L.lphv()) == 0)
        a.lse[(int64_t)r * a.heads + L.head] = st.s > 0.f ? (st.m + log2f(st.s)) * kLn2 : -INFINITY;
}

// Destination-side data of row r: GATv2 l_r (unpacked) and A_l[r, head];
// GT Q_r pre-scaled by scale * log2 e.
template <int KIND, class T, int CPL, int LPH>
__device__ __forceinline__ void load_dest(const AttnArgs &a, const Lane<KIND, T, CPL, LPH> &L, int32_t r,
                                          float *dq, float *al) {
    constexpr int NC = CPL * Elt<T>::N;
    const char *row = a.Qd + (int64_t)r * a.qd_stride;
    uint4 v[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
        v[c] = L.act() ? ldg16(row + (L.lane * CPL + c) * 16) : make_uint4(0u, 0u, 0u, 0u);
    unpack_row<T, CPL>(v, dq);
    if (KIND == ATT_GT) {
#pragma unroll
        for (int k = 0; k < NC; ++k) dq[k] *= a.qscale;
        *al = 0.f;
    } else {
        *al = L.act() ? __ldg(reinterpret_cast<const float *>(row + a.ar_off) + L.head) : 0.f;
    }
}

// A piece of heavy row r (edges of run w) leaves its state in slot 2w+1 (the
// row's first piece) or 2w (a later piece); the last piece to arrive merges
// the pieces of runs wa..wb in order and writes the row.
template <int KIND, class T, int CPL, int LPH>
__device__ __forceinline__ void flush_piece(const AttnArgs &a, const Lane<KIND, T, CPL, LPH> &L, int64_t w,
                                            int32_t r, const SmState<CPL * Elt<T>::N> &st) {
    constexpr int NC = CPL * Elt<T>::N;
    const int64_t stride = slot_stride(a.HD, a.heads);
    const int32_t rb = __ldg(a.rowptr + r), re = __ldg(a.rowptr + r + 1);
    const int64_t E = kAttnE;
    const int64_t wa = rb / E, wb = ((int64_t)re - 1) / E;
    float *slot = a.slots + (2 * w + (w == wa ? 1 : 0)) * stride;
    if (L.act()) {
#pragma unroll
        for (int k = 0; k < NC; k += 4)
            __stcg(reinterpret_cast<float4 *>(slot + L.lane * NC + k),
                   make_float4(st.acc[k], st.acc[k + 1], st.acc[k + 2], st.acc[k + 3]));
        if ((L.lane % L.lphv()) == 0) {
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
        const float mk = L.act() ? __ldcg(sk + a.HD + 2 * L.head) : -INFINITY;
        const float sk_s = L.act() ? __ldcg(sk + a.HD + 2 * L.head + 1) : 0.f;
        const float mx = fmaxf(m.m, mk);
        const float c_old = (m.m == -INFINITY) ? 0.f : exp2f(m.m - mx);
        const float c_new = (mk == -INFINITY) ? 0.f : exp2f(mk - mx);
        m.s = m.s * c_old + sk_s * c_new;
        if (L.act()) {
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
    store_final<KIND, T, CPL, LPH>(a, L, r, m);
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

// The warp's edge stream: edges [sb, se) in batches of U through S stages.
struct Ring {
    unsigned char *stages;  // S * U * rec bytes
    uint64_t *bars;         // S mbarriers
    int32_t sb, se, nb;     // span and its batch count
    int32_t k_issue;        // next batch to issue
    int32_t kc;             // batch of the next edge to consume
    int32_t cs;             // its stage (kc mod S)
    uint32_t cph;           // its mbarrier phase parity ((kc / S) mod 2)
    int32_t u;              // position of that edge in its batch
    bool ready;             // batch kc has been waited for
    int32_t pcol;           // prefetched column id of lane's edge in batch k_issue
    bool bail;
};

// Issue batch R.k_issue into stage st (the stage batch k_issue - S used).
template <int KIND, class T, int CPL, int LPH>
__device__ __forceinline__ void ring_issue(const AttnArgs &a, Ring &R, int lane, int32_t st) {
    using Gm = Geo<KIND, T, CPL, LPH>;
    const int32_t k = R.k_issue;
    const int32_t base = R.sb + k * Gm::U(a);
    const int32_t cnt = min(Gm::U(a), R.se - base);
    uint64_t *bar = R.bars + st;
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)(cnt * (Gm::s_bytes(a) + Gm::v_bytes(a))));
    __syncwarp();
    if (lane < cnt) {
        unsigned char *dst = R.stages + ((size_t)st * Gm::U(a) + lane) * Gm::rec(a);
        const int64_t j = R.pcol;
        bulk_g2s(dst, a.Sg + j * a.sg_stride, (uint32_t)Gm::s_bytes(a), bar);
        if (Gm::v_bytes(a)) bulk_g2s(dst + Gm::s_bytes(a), a.Vg + j * a.vg_stride, (uint32_t)Gm::v_bytes(a), bar);
    }
    const int32_t nxt = base + Gm::U(a) + lane;
    R.pcol = (lane < Gm::U(a) && nxt < R.se) ? __ldg(a.colidx + nxt) : 0;
    ++R.k_issue;
}

// Fold the edges [b, end) of the span (consecutive with what was consumed
// before) into st.
template <int KIND, class T, int CPL, int LPH>
__device__ __forceinline__ void consume(const AttnArgs &a, const Lane<KIND, T, CPL, LPH> &L, Ring &R, int32_t b,
                                        int32_t end, const float *dq, float al, SmState<CPL * Elt<T>::N> &st) {
    using Gm = Geo<KIND, T, CPL, LPH>;
    int32_t e = b;
    while (e < end && !R.bail) {
        if (!R.ready) {
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(R.bars + R.cs, R.cph));
            if (!ok) {
                set_device_error(a.err, GNN_ERR_TIMEOUT);
                R.bail = true;
                return;
            }
            R.ready = true;
        }
        const unsigned char *stage = R.stages + (size_t)R.cs * Gm::U(a) * Gm::rec(a);
        const int32_t n = min(Gm::U(a) - R.u, end - e);
        int32_t g = 0;
        constexpr int NG = att_group(KIND, CPL * Elt<T>::N);
        for (; g + NG <= n; g += NG)
            fold_edges<KIND, T, CPL, LPH, NG>(a, L, stage + (size_t)(R.u + g) * Gm::rec(a), dq, al, st);
        for (; g < n; ++g) fold_edges<KIND, T, CPL, LPH, 1>(a, L, stage + (size_t)(R.u + g) * Gm::rec(a), dq, al, st);
        e += n;
        R.u += n;
        if (R.u == Gm::U(a) || e == R.se) {
            // batch consumed: its stage takes the batch S ahead
            __syncwarp();
            fence_proxy_async_smem();
            if (R.k_issue < R.nb) ring_issue<KIND, T, CPL, LPH>(a, R, L.lane, R.cs);
            ++R.kc;
            if (++R.cs == Gm::S(a)) {
                R.cs = 0;
                R.cph ^= 1u;
            }
            R.u = 0;
            R.ready = false;
        }
    }
}

template <int KIND, class T, int CPL, int LPH>
__global__ void __launch_bounds__(kAttnWarps * 32, att_min_blocks(KIND, CPL * Elt<T>::N)) k_attn(AttnArgs a) {
    constexpr int NC = CPL * Elt<T>::N;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int64_t w = (int64_t)blockIdx.x * kAttnWarps + warp;
    if (w >= a.n_workers) return;
    Lane<KIND, T, CPL, LPH> L;
    L.lane = threadIdx.x & 31;
    L.active = L.lane * CPL < a.nch;
    L.lph = a.D / NC;
    L.head = L.act() ? (L.lane * NC) / a.D : 0;
    if (KIND == ATT_GATV2) {
#pragma unroll
        for (int k = 0; k < NC; ++k) L.coef[k] = L.act() ? __ldg(a.coef + L.lane * NC + k) : 0.f;
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
    // a heavy row that started in an earlier run and reaches into this one
    int32_t h = -1, lo_beg = 0;
    if (lo > 0 && e0 < a.nnz) {
        lo_beg = __ldg(rowptr + lo);
        if (lo_beg > e0 && lo_beg - __ldg(rowptr + lo - 1) > E) h = lo - 1;
    }
    // the span of edges this warp folds
    Ring R;
    R.sb = h >= 0 ? (int32_t)e0 : (lo < lo_end ? __ldg(rowptr + lo) : 0);
    if (lo < lo_end) {
        const int32_t rl = lo_end - 1;
        const int32_t rlb = __ldg(rowptr + rl), rle = __ldg(rowptr + rl + 1);
        R.se = (rle - rlb > E) ? (int32_t)e1 : rle;
    } else {
        R.se = h >= 0 ? (int32_t)min((int64_t)lo_beg, e1) : R.sb;
    }
    using Gm = Geo<KIND, T, CPL, LPH>;
    R.nb = (R.se - R.sb + Gm::U(a) - 1) / Gm::U(a);
    R.stages = smem + (size_t)warp * a.ring_bytes;
    R.bars = reinterpret_cast<uint64_t *>(R.stages + (size_t)Gm::S(a) * Gm::U(a) * Gm::rec(a));
    R.k_issue = 0;
    R.kc = 0;
    R.cs = 0;
    R.cph = 0;
    R.u = 0;
    R.ready = false;
    R.bail = false;
    R.pcol = 0;
    if (R.nb > 0) {
        if (L.lane == 0) {
            for (int s = 0; s < Gm::S(a); ++s) mbar_init(R.bars + s, 1);
            mbar_init_fence();
        }
        __syncwarp();
        R.pcol = (L.lane < Gm::U(a) && R.sb + L.lane < R.se) ? __ldg(a.colidx + R.sb + L.lane) : 0;
        for (int s = 0; s < Gm::S(a) && R.k_issue < R.nb; ++s) ring_issue<KIND, T, CPL, LPH>(a, R, L.lane, s);
    }

    float dq[NC];
    float al;
    SmState<NC> st;
    if (h >= 0) {
        load_dest<KIND, T, CPL, LPH>(a, L, h, dq, &al);
        st.reset();
        consume<KIND, T, CPL, LPH>(a, L, R, R.sb, (int32_t)min((int64_t)lo_beg, e1), dq, al, st);
        if (!R.bail) flush_piece<KIND, T, CPL, LPH>(a, L, w, h, st);
    }
    // owned rows, 32 at a time: lanes read the bounds of 32 rows and only the
    // non-empty ones are visited (empty rows are written by k_attn_empty_rows)
    for (int32_t rbase = lo; rbase < lo_end && !R.bail; rbase += 32) {
        const int32_t rr = rbase + L.lane;
        int32_t my_b = 0, my_e = 0;
        if (rr < lo_end) {
            my_b = __ldg(rowptr + rr);
            my_e = __ldg(rowptr + rr + 1);
        }
        unsigned todo = __ballot_sync(0xffffffffu, my_e > my_b);
        while (todo && !R.bail) {
            const int k = __ffs(todo) - 1;
            todo &= todo - 1;
            const int32_t r = rbase + k;
            const int32_t rb = __shfl_sync(0xffffffffu, my_b, k), re = __shfl_sync(0xffffffffu, my_e, k);
            st.reset();
            load_dest<KIND, T, CPL, LPH>(a, L, r, dq, &al);
            if (re - rb > E) {  // heavy: this run holds its first piece (and it is the last owned row)
                consume<KIND, T, CPL, LPH>(a, L, R, rb, (int32_t)e1, dq, al, st);
                if (!R.bail) flush_piece<KIND, T, CPL, LPH>(a, L, w, r, st);
            } else {
                consume<KIND, T, CPL, LPH>(a, L, R, rb, re, dq, al, st);
                store_final<KIND, T, CPL, LPH>(a, L, r, st);
            }
        }
    }
    if (R.bail) {
        // let the copies still in flight land before the warp leaves
        for (int32_t k = R.kc; k < R.k_issue; ++k) mbar_wait_bounded(R.bars + (k % Gm::S(a)), (uint32_t)((k / Gm::S(a)) & 1u));
    }
}

// Rows without edges: out = 0, lse = -inf (one thread per row and head).
__global__ void k_attn_empty_rows(const int32_t *__restrict__ rowptr, int32_t n_rows, int32_t HD, int32_t heads,
                                  float *__restrict__ out, float *__restrict__ lse) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)n_rows * heads) return;
    const int32_t r = (int32_t)(i / heads), h = (int32_t)(i % heads);
    if (rowptr[r + 1] != rowptr[r]) return;
    const int32_t D = HD / heads;
    float *o = out + (int64_t)r * HD + (int64_t)h * D;
    for (int32_t d = 0; d < D; d += 4) *reinterpret_cast<float4 *>(o + d) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse) lse[i] = -INFINITY;
}

// GATv2 per-node linear parts: A[i,h] = sum_d lin[hD+d] C[i, hD+d], written
// into the padding of the projected row.  One warp per node.
template <class T>
__global__ void __launch_bounds__(256) k_gatv2_linear(char *__restrict__ C, int64_t row_bytes, int64_t n,
                                                      int32_t heads, int32_t D, const float *__restrict__ lin) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= n) return;
    const T *row = reinterpret_cast<const T *>(C + i * row_bytes);
    float *A = reinterpret_cast<float *>(C + i * row_bytes + (int64_t)heads * D * sizeof(T));
    for (int32_t h = 0; h < heads; ++h) {
        float s = 0.f;
        for (int32_t d = lane; d < D; d += 32) {
            float c;
            if constexpr (sizeof(T) == 4) c = (float)row[h * D + d];
            else c = __bfloat162float(row[h * D + d]);
            s = fmaf(__ldg(lin + h * D + d), c, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) A[h] = s;
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
// C[n, Fo] = H[n, Fi] W[Fi, Fo] (C rows ldc elements apart), fp32 FMA (no
// TF32), output in T (bf16 by round-to-nearest-even).  64x64 tile per
// 256-thread block, 4x4 per thread.
template <class T>
__global__ void __launch_bounds__(256) k_proj_simt(const T *__restrict__ H, const T *__restrict__ W,
                                                   T *__restrict__ C, int64_t n, int32_t Fi, int32_t Fo,
                                                   int64_t ldc) {
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
            if constexpr (sizeof(T) == 4) C[gr * ldc + gc] = acc[p][q];
            else C[gr * ldc + gc] = __float2bfloat16_rn(acc[p][q]);
        }
    }
}

}  // namespace

// tcgen05 projection (bf16), defined in projection.cu; returns
// GNN_ERR_UNSUPPORTED for shapes it does not cover.  ldc: C row stride in
// elements; lin_out/lin_ld: per-node linear parts and their row stride in
// floats.
gnn_status projection_tc_lin(const void *H, int64_t n, int32_t Fi, const void *W, int32_t Fo, void *C,
                             int64_t ldc, const float *lin_coef, int32_t heads, int32_t D, float *lin_out,
                             int64_t lin_ld, cudaStream_t s);

static gnn_status projection_simt(const void *H, int32_t dtype, int64_t n, int32_t F_in, const void *W,
                                  int32_t F_out, void *C, int64_t ldc, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    dim3 grid((unsigned)((n + 63) / 64), (unsigned)((F_out + 63) / 64));
    if (dtype == GNN_F32)
        k_proj_simt<float><<<grid, 256, 0, s>>>(static_cast<const float *>(H), static_cast<const float *>(W),
                                                 static_cast<float *>(C), n, F_in, F_out, ldc);
    else
        k_proj_simt<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(H),
                                                         static_cast<const __nv_bfloat16 *>(W),
                                                         static_cast<__nv_bfloat16 *>(C), n, F_in, F_out, ldc);
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
    char *l, *r;  // padded projected rows [n, gat_row_bytes]
    float *coef, *lin, *slots;
    int32_t *tickets;
    int64_t row_bytes;
    size_t bytes;
};

static GatLayout gat_layout(const gnn_csr *g, void *base, int32_t esize, bool separate, int32_t heads,
                            int32_t head_dim) {
    Carver c(base);
    GatLayout L;
    const int32_t HD = heads * head_dim;
    const int64_t nw = attn_workers(g);
    L.row_bytes = gat_row_bytes(HD, heads, esize);
    L.l = c.take<char>((size_t)g->n_cols * L.row_bytes);
    L.r = separate ? c.take<char>((size_t)g->n_cols * L.row_bytes) : L.l;
    L.coef = c.take<float>(HD);
    L.lin = c.take<float>(HD);
    L.slots = c.take<float>((size_t)2 * nw * (size_t)slot_stride(HD, heads));
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

// Ring geometry: two stages of U records per warp.  Measured on GB300 (GT,
// 1 KB records: U = 4; GATv2, 528-byte records: U = 8): deeper rings cost
// more shared memory per warp than they gain, since fewer warps fit.
static void ring_shape(AttnArgs &a) {
    a.rec = a.s_bytes + a.v_bytes;
    a.U = a.rec <= 640 ? 8 : 4;
    a.S = 2;
    a.ring_bytes = (int32_t)round_up((size_t)a.S * a.U * a.rec + (size_t)a.S * 8, 128);
}

template <int KIND, class T, int CPL, int LPH>
static cudaError_t launch_attn_lph(const AttnArgs &a, cudaStream_t s) {
    const cudaError_t attr = func_attr(reinterpret_cast<const void *>(k_attn<KIND, T, CPL, LPH>),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (attr != cudaSuccess) return attr;
    if (!Geo<KIND, T, CPL, LPH>::agrees(a)) return cudaErrorInvalidValue;
    const size_t smem = (size_t)kAttnWarps * a.ring_bytes;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    const int blocks = (int)((a.n_workers + kAttnWarps - 1) / kAttnWarps);
    k_attn<KIND, T, CPL, LPH><<<blocks, kAttnWarps * 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <int KIND, class T>
static cudaError_t launch_attn(const AttnArgs &a, int cpl, cudaStream_t s) {
    if constexpr (sizeof(T) == 2) {
        // bf16: at most 256 channels, one chunk per lane; a compile-time
        // lanes-per-head (D/8) when all 32 lanes own channels
        if (a.nch != 32) return launch_attn_lph<KIND, T, 1, 0>(a, s);
        switch (a.D / 8) {
            case 4: return launch_attn_lph<KIND, T, 1, 4>(a, s);
            case 8: return launch_attn_lph<KIND, T, 1, 8>(a, s);
            default: return launch_attn_lph<KIND, T, 1, 16>(a, s);
        }
    } else {
        switch (cpl) {
            case 1: return launch_attn_lph<KIND, T, 1, 0>(a, s);
            case 2: return launch_attn_lph<KIND, T, 2, 0>(a, s);
            case 4: return launch_attn_lph<KIND, T, 4, 0>(a, s);
            default: return launch_attn_lph<KIND, T, 8, 0>(a, s);
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
    if (n == 0) return GNN_OK;
    cudaStream_t s = as_stream(stream);
    if (dtype == GNN_BF16) {
        gnn_status st = projection_tc_lin(H, n, F_in, W, F_out, C, F_out, nullptr, 0, 0, nullptr, 0, s);
        if (st != GNN_ERR_UNSUPPORTED) return st;
    }
    return projection_simt(H, dtype, n, F_in, W, F_out, C, F_out, s);
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
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    const int32_t HD = heads * head_dim;
    const int64_t n = g->n_cols;

    // coefficients of the |.| part and of the per-node linear parts
    const float half_1ps = 0.5f * (1.f + neg_slope), half_1ms = 0.5f * (1.f - neg_slope);
    k_gatv2_coef<<<(HD + 255) / 256, 256, 0, s>>>(a, HD, half_1ms, half_1ps, WL.coef, WL.lin);
    note_launch();
    GNN_LAUNCH_CHECK();
    // a3: projections l = H W_l (and r = H W_r) into padded rows, with the
    // linear parts A_l, A_r in the padding
    const void *Ws[2] = {W_l, W_r};
    char *Cs[2] = {WL.l, WL.r};
    const int64_t ldc = WL.row_bytes / esize;
    for (int k = 0; k < (separate ? 2 : 1); ++k) {
        float *A = reinterpret_cast<float *>(Cs[k] + (int64_t)HD * esize);
        st = GNN_ERR_UNSUPPORTED;
        if (dtype == GNN_BF16)
            st = projection_tc_lin(H, n, F_in, Ws[k], HD, Cs[k], ldc, WL.lin, heads, head_dim, A,
                                   WL.row_bytes / 4, s);
        if (st == GNN_ERR_UNSUPPORTED) {
            st = projection_simt(H, dtype, n, F_in, Ws[k], HD, Cs[k], ldc, s);
            if (st != GNN_OK) return st;
            const int lin_blocks = (int)((n * 32 + 255) / 256);
            if (dtype == GNN_F32)
                k_gatv2_linear<float><<<lin_blocks, 256, 0, s>>>(Cs[k], WL.row_bytes, n, heads, head_dim, WL.lin);
            else
                k_gatv2_linear<__nv_bfloat16><<<lin_blocks, 256, 0, s>>>(Cs[k], WL.row_bytes, n, heads, head_dim,
                                                                          WL.lin);
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
    A.Sg = WL.r;
    A.Vg = nullptr;
    A.Qd = WL.l;
    A.sg_stride = A.qd_stride = WL.row_bytes;
    A.vg_stride = 0;
    A.s_bytes = (int32_t)WL.row_bytes;
    A.v_bytes = 0;
    A.ar_off = HD * esize;
    A.coef = WL.coef;
    A.out = out;
    A.lse = lse;
    A.slots = WL.slots;
    A.tickets = WL.tickets;
    A.err = err;
    A.nnz = g->nnz;
    A.n_workers = attn_workers(g);
    A.n_rows = g->n_rows;
    A.HD = HD;
    A.heads = heads;
    A.D = head_dim;
    A.nch = nch;
    ring_shape(A);
    k_attn_empty_rows<<<(int)(((int64_t)g->n_rows * heads + 255) / 256), 256, 0, s>>>(g->rowptr, g->n_rows, HD,
                                                                                      heads, out, lse);
    note_launch();
    if (g->nnz == 0) {
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }
    cudaError_t e = dtype == GNN_F32 ? launch_attn<ATT_GATV2, float>(A, cpl, s)
                                     : launch_attn<ATT_GATV2, __nv_bfloat16>(A, cpl, s);
    note_launch();
    if (e != cudaSuccess) return cuda_status(e);
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
    int32_t *err = device_error_word();
    if (!err) return GNN_ERR_CUDA;
    const int32_t esize = dtype == GNN_F32 ? 4 : 2;
    Carver cv(ws);
    AttnArgs A{};
    A.rowptr = g->rowptr;
    A.colidx = g->colidx;
    A.run_table = prep ? prep_run_table(g, prep) : nullptr;
    A.Sg = static_cast<const char *>(K);
    A.Vg = static_cast<const char *>(V);
    A.Qd = static_cast<const char *>(Q);
    A.sg_stride = A.vg_stride = A.qd_stride = (int64_t)heads * head_dim * esize;
    A.s_bytes = A.v_bytes = heads * head_dim * esize;
    A.ar_off = 0;
    A.qscale = scale * kLog2e;
    A.out = out;
    A.lse = lse;
    A.err = err;
    A.n_workers = attn_workers(g);
    A.slots = cv.take<float>((size_t)2 * A.n_workers * (size_t)slot_stride(heads * head_dim, heads));
    A.tickets = cv.take<int32_t>((size_t)A.n_workers);
    A.nnz = g->nnz;
    A.n_rows = g->n_rows;
    A.HD = heads * head_dim;
    A.heads = heads;
    A.D = head_dim;
    A.nch = nch;
    ring_shape(A);
    k_attn_empty_rows<<<(int)(((int64_t)g->n_rows * heads + 255) / 256), 256, 0, s>>>(g->rowptr, g->n_rows,
                                                                                      A.HD, heads, out, lse);
    note_launch();
    if (g->nnz == 0) {
        GNN_LAUNCH_CHECK();
        return GNN_OK;
    }
    cudaError_t e = dtype == GNN_F32 ? launch_attn<ATT_GT, float>(A, cpl, s)
                                     : launch_attn<ATT_GT, __nv_bfloat16>(A, cpl, s);
    note_launch();
    if (e != cudaSuccess) return cuda_status(e);
    return GNN_OK;
}

}  // extern "C"
