/*
 * CPU oracle for CSR neighbourhood aggregation -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
 * leg may load or call this library.  The CUDA library never does, and this
 * file shares no code, header or constant table with it.
 *
 * Plain, slow, single-threaded definitions with fp64 accumulation.  Inputs
 * are fp32, or bf16 given as raw 16-bit patterns (dtype 1), widened exactly.
 * The source paper is "On efficient scaling of GNNs via IO-aware layer
 * implementations" (cited below as "IO-aware GNN layers"); the reordering
 * follows "A High-Throughput Solver for Marginalized Graph Kernels on GPU"
 * (Section on reordering, RCM).
 *
 * Graph convention: CSR by destination -- row i lists the sources j of the
 * edges j -> i, so N(i) = colidx[rowptr[i] .. rowptr[i+1]).
 *
 * Every function below is pinned by CPU tests (dense brute force, closed
 * forms, invariants); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR 1

static double widen(const void *p, int dtype, int64_t i) {
    if (dtype == 0) return (double)((const float *)p)[i];
    uint32_t u = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static int32_t sel_row(const int32_t *rows, int32_t s) { return rows ? rows[s] : s; }

/* ------------------------------------------------------------------ */
/* degrees                                                             */
/* ------------------------------------------------------------------ */

/* d_in(i) = length of row i; d_out(j) = occurrences of j among all columns
 * (self-loops included in both). */
int orc_degrees(int32_t n_rows, int32_t n_cols, const int32_t *rowptr,
                const int32_t *colidx, int32_t *d_in, int32_t *d_out) {
    for (int32_t i = 0; i < n_rows; ++i) d_in[i] = rowptr[i + 1] - rowptr[i];
    for (int32_t j = 0; j < n_cols; ++j) d_out[j] = 0;
    for (int64_t e = 0; e < rowptr[n_rows]; ++e) {
        int32_t j = colidx[e];
        if (j < 0 || j >= n_cols) return ORC_ERR;
        d_out[j]++;
    }
    return ORC_OK;
}

/* Degree statistics of the row lengths d_i = rowptr[i+1] - rowptr[i] (the
 * in-degrees), the graph statistics an adaptive choice of backend reads
 * (IO-aware GNN layers, Section 5, degree skew; Appendix B.1, Table 5's
 * skewness): out = {mean, standard deviation, skewness, max}, population
 * moments from two passes: mean = sum d / n, m_k = sum (d - mean)^k / n,
 * std = sqrt(m_2), skewness = m_3 / m_2^(3/2) (0 when m_2 = 0). */
int orc_degree_stats(int32_t n, const int32_t *rowptr, double *out) {
    out[0] = out[1] = out[2] = out[3] = 0.0;
    if (n <= 0) return ORC_OK;
    double sum = 0.0, mx = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        double d = (double)(rowptr[i + 1] - rowptr[i]);
        sum += d;
        if (d > mx) mx = d;
    }
    double mean = sum / n, m2 = 0.0, m3 = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        double c = (double)(rowptr[i + 1] - rowptr[i]) - mean;
        m2 += c * c;
        m3 += c * c * c;
    }
    m2 /= n;
    m3 /= n;
    out[0] = mean;
    out[1] = sqrt(m2);
    out[2] = m2 > 0.0 ? m3 / (m2 * sqrt(m2)) : 0.0;
    out[3] = mx;
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* SpMM  (IO-aware GNN layers, Section 2.2 (i); Appendix D.4)          */
/* ------------------------------------------------------------------ */

/*
 * Y[i,:] = sum_{e in row i} w_e * X[colidx[e], :]
 * w_e = values[e] (or 1 when values is NULL) times the normalisation factor:
 *   norm 0 none:  1
 *   norm 1 left:  1 / d_in(i)
 *   norm 2 right: 1 / d_out(j)
 *   norm 3 both:  1 / sqrt(d_in(i) * d_out(j))     (GCN, Kipf & Welling)
 * Rows with no edges give 0.  Only the selected rows are computed
 * (rows == NULL: all rows, n_sel = n_rows); Y is [n_sel, F].
 */
int orc_spmm(int32_t n_rows, int32_t n_cols, const int32_t *rowptr,
             const int32_t *colidx, const float *values, int norm,
             const void *X, int dtype, int32_t F, const int32_t *rows,
             int32_t n_sel, double *Y) {
    int32_t *d_out = NULL;
    if (norm == 2 || norm == 3) {
        d_out = calloc((size_t)n_cols, sizeof(int32_t));
        if (!d_out) return ORC_ERR;
        for (int64_t e = 0; e < rowptr[n_rows]; ++e) d_out[colidx[e]]++;
    }
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        double *y = Y + (int64_t)s * F;
        for (int32_t f = 0; f < F; ++f) y[f] = 0.0;
        int64_t d_in = rowptr[i + 1] - rowptr[i];
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
            int32_t j = colidx[e];
            double w = values ? (double)values[e] : 1.0;
            if (norm == 1) w /= (double)d_in;
            else if (norm == 2) w /= (double)d_out[j];
            else if (norm == 3) w /= sqrt((double)d_in * (double)d_out[j]);
            for (int32_t f = 0; f < F; ++f)
                y[f] += w * widen(X, dtype, (int64_t)j * F + f);
        }
    }
    free(d_out);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* segment reductions (IO-aware GNN layers, Section 2.2 (ii); D.1)     */
/* ------------------------------------------------------------------ */

/* Order-preserving 32-bit key of an fp32 value (IO-aware GNN layers,
 * Appendix D.1, order-preserving packing for atomic reductions): negative
 * values have every bit inverted, non-negative values get the sign bit set,
 * so unsigned comparison of keys orders the floats (and -0 < +0). */
uint32_t orc_order_key(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/*
 * op 0 sum, 1 mean (= sum / d_in(i)), 2 max, 3 min.
 * max: the neighbour value with the largest order key; among equal keys the
 * smallest source node id wins; argmax[s,f] = that source node id.
 * min (IO-aware GNN layers, Appendix D.1: the min reduction with its argmin,
 * values compared through the order-preserving key and ties resolved by the
 * source index): the neighbour value with the smallest order key, the
 * smallest source id among equal keys; argmin[s,f] = that id.
 * A row with no edges gives 0 (and arg -1).  Y is [n_sel, F].
 */
int orc_segment_reduce(int op, int32_t n_rows, const int32_t *rowptr,
                       const int32_t *colidx, const void *X, int dtype,
                       int32_t F, const int32_t *rows, int32_t n_sel, double *Y,
                       int32_t *argmax) {
    (void)n_rows;
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        int64_t b = rowptr[i], e_end = rowptr[i + 1];
        for (int32_t f = 0; f < F; ++f) {
            double acc = 0.0;
            int32_t best_j = -1;
            uint32_t best_key = 0;
            double best_v = 0.0;
            for (int64_t e = b; e < e_end; ++e) {
                int32_t j = colidx[e];
                double v = widen(X, dtype, (int64_t)j * F + f);
                if (op == 2 || op == 3) {
                    uint32_t k = orc_order_key((float)v);
                    int better = (op == 2) ? (k > best_key) : (k < best_key);
                    if (best_j < 0 || better || (k == best_key && j < best_j)) {
                        best_key = k;
                        best_j = j;
                        best_v = v;
                    }
                } else {
                    acc += v;
                }
            }
            double out;
            if (op == 0) out = acc;
            else if (op == 1) out = (e_end > b) ? acc / (double)(e_end - b) : 0.0;
            else out = (best_j >= 0) ? best_v : 0.0;
            Y[(int64_t)s * F + f] = out;
            if ((op == 2 || op == 3) && argmax) argmax[(int64_t)s * F + f] = best_j;
        }
    }
    return ORC_OK;
}

/*
 * CSR^T (the transpose the backward kernels of IO-aware GNN layers,
 * Appendix D.2, run over): row j of the result lists every i with j in
 * N(i), in ascending i, with that edge's value.  rowptr_t [n_cols + 1],
 * colidx_t and values_t (may be NULL) [nnz].
 */
int orc_csr_transpose(int32_t n_rows, int32_t n_cols, const int32_t *rowptr, const int32_t *colidx,
                      const float *values, int32_t *rowptr_t, int32_t *colidx_t, float *values_t) {
    for (int32_t j = 0; j <= n_cols; ++j) rowptr_t[j] = 0;
    for (int32_t i = 0; i < n_rows; ++i)
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
            if (colidx[e] < 0 || colidx[e] >= n_cols) return ORC_ERR;
            rowptr_t[colidx[e] + 1] += 1;
        }
    for (int32_t j = 0; j < n_cols; ++j) rowptr_t[j + 1] += rowptr_t[j];
    /* fill row by row in ascending i: each transposed row comes out sorted */
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_cols > 0 ? n_cols : 1));
    if (!next) return ORC_ERR;
    for (int32_t j = 0; j < n_cols; ++j) next[j] = rowptr_t[j];
    for (int32_t i = 0; i < n_rows; ++i)
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
            int32_t k = next[colidx[e]]++;
            colidx_t[k] = i;
            if (values_t) values_t[k] = values ? values[e] : 1.0f;
        }
    free(next);
    return ORC_OK;
}

/*
 * Backward of the max / min reduction (IO-aware GNN layers, Appendix D.1,
 * the backward pass as a sparse scatter through the stored argmin): the
 * gradient of out[v,f] flows only to the selected source, so
 *   grad_X[j,f] = sum over v with arg[v,f] == j of grad_out[v,f]
 * (arg -1, an empty row, contributes nothing).  arg and grad_out are
 * [n_rows, F]; grad_X is [n_cols, F], fp64, overwritten.
 */
int orc_reduce_ext_backward(int32_t n_rows, int32_t n_cols, int32_t F, const int32_t *arg,
                            const double *grad_out, double *grad_X) {
    for (int64_t k = 0; k < (int64_t)n_cols * F; ++k) grad_X[k] = 0.0;
    for (int32_t v = 0; v < n_rows; ++v)
        for (int32_t f = 0; f < F; ++f) {
            int32_t j = arg[(int64_t)v * F + f];
            if (j < 0) continue;
            if (j >= n_cols) return ORC_ERR;
            grad_X[(int64_t)j * F + f] += grad_out[(int64_t)v * F + f];
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* attention (IO-aware GNN layers, Section 2.2 (iii); Appendix D.2)    */
/* ------------------------------------------------------------------ */

/* softmax over the logits e[0..deg) of one (row, head); writes alpha and
 * returns logsumexp = m + ln sum exp(e - m) (natural log). */
static double softmax_row(const double *e, int64_t deg, double *alpha) {
    if (deg == 0) return -INFINITY;
    double m = e[0];
    for (int64_t k = 1; k < deg; ++k)
        if (e[k] > m) m = e[k];
    double s = 0.0;
    for (int64_t k = 0; k < deg; ++k) s += exp(e[k] - m);
    for (int64_t k = 0; k < deg; ++k) alpha[k] = exp(e[k] - m) / s;
    return m + log(s);
}

/* row i of C = H * W (H [., F_in], W [F_in, HD] row-major), in fp64 */
static void project_row(const void *H, int dtype, int32_t F_in, const void *W,
                        int32_t HD, int32_t i, double *out) {
    for (int32_t c = 0; c < HD; ++c) out[c] = 0.0;
    for (int32_t k = 0; k < F_in; ++k) {
        double h = widen(H, dtype, (int64_t)i * F_in + k);
        for (int32_t c = 0; c < HD; ++c) out[c] += h * widen(W, dtype, (int64_t)k * HD + c);
    }
}

/*
 * GATv2 forward for the selected destination rows i, every head h:
 *   l_i = H_i W_l,  r_j = H_j W_r        (W_r NULL: W_r = W_l)
 *   e_ij = sum_d a[h,d] * LeakyReLU_slope(l_i[h,d] + r_j[h,d])
 *   alpha_ij = softmax over j in N(i) of e_ij
 *   out_i[h,:] = sum_j alpha_ij r_j[h,:],  lse[i,h] = ln sum_j exp(e_ij)
 * Head h owns columns [h*D, (h+1)*D).  out [n_sel, heads*D], lse [n_sel,
 * heads]; alpha (optional) [edges of the selected rows in order, heads].
 */
/* x rounded to the nearest fp32 and then to the nearest bf16 (ties to
 * even on the fp32 bits), returned widened: the storage rounding of the
 * projected features in the bf16 path (IO-aware GNN layers, Section 2.2
 * (iii): attention logits computed on projected features). */
static double round_bf16(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    memcpy(&f, &u, 4);
    return (double)f;
}

static void round_bf16_all(double *v, int64_t n) {
    for (int64_t k = 0; k < n; ++k) v[k] = round_bf16(v[k]);
}

int orc_gatv2_ex(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
                 const void *H, int dtype, int32_t F_in, const void *W_l,
                 const void *W_r, const float *a, int32_t heads, int32_t D,
                 double slope, const int32_t *rows, int32_t n_sel, int round_c,
                 double *out, double *lse, double *alpha);

int orc_gatv2(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
              const void *H, int dtype, int32_t F_in, const void *W_l,
              const void *W_r, const float *a, int32_t heads, int32_t D,
              double slope, const int32_t *rows, int32_t n_sel, double *out,
              double *lse, double *alpha) {
    return orc_gatv2_ex(n_rows, rowptr, colidx, H, dtype, F_in, W_l, W_r, a, heads, D, slope,
                        rows, n_sel, 0, out, lse, alpha);
}

/* As orc_gatv2; round_c != 0 is the diagnostic mode: every projected
 * feature l_i and r_j is rounded to bf16 before the attention, as the bf16
 * path stores them, so what remains between a kernel and this result is the
 * kernel's own arithmetic. */
int orc_gatv2_ex(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
                 const void *H, int dtype, int32_t F_in, const void *W_l,
                 const void *W_r, const float *a, int32_t heads, int32_t D,
                 double slope, const int32_t *rows, int32_t n_sel, int round_c,
                 double *out, double *lse, double *alpha) {
    (void)n_rows;
    int32_t HD = heads * D;
    if (!W_r) W_r = W_l;
    int64_t max_deg = 0;
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        int64_t d = rowptr[i + 1] - rowptr[i];
        if (d > max_deg) max_deg = d;
    }
    double *l = malloc(sizeof(double) * (size_t)HD);
    double *R = malloc(sizeof(double) * (size_t)HD * (size_t)(max_deg > 0 ? max_deg : 1));
    double *e = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double *al = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    if (!l || !R || !e || !al) { free(l); free(R); free(e); free(al); return ORC_ERR; }
    int64_t alpha_pos = 0;
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        int64_t b = rowptr[i], deg = rowptr[i + 1] - b;
        project_row(H, dtype, F_in, W_l, HD, i, l);
        for (int64_t k = 0; k < deg; ++k)
            project_row(H, dtype, F_in, W_r, HD, colidx[b + k], R + k * HD);
        if (round_c) {
            round_bf16_all(l, HD);
            round_bf16_all(R, deg * HD);
        }
        for (int32_t h = 0; h < heads; ++h) {
            for (int64_t k = 0; k < deg; ++k) {
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d) {
                    double x = l[h * D + d] + R[k * HD + h * D + d];
                    double act = x > 0.0 ? x : slope * x;
                    acc += (double)a[h * D + d] * act;
                }
                e[k] = acc;
            }
            double L = softmax_row(e, deg, al);
            lse[(int64_t)s * heads + h] = L;
            for (int32_t d = 0; d < D; ++d) {
                double o = 0.0;
                for (int64_t k = 0; k < deg; ++k) o += al[k] * R[k * HD + h * D + d];
                out[(int64_t)s * HD + h * D + d] = o;
            }
            if (alpha)
                for (int64_t k = 0; k < deg; ++k) alpha[(alpha_pos + k) * heads + h] = al[k];
        }
        alpha_pos += deg;
    }
    free(l); free(R); free(e); free(al);
    return ORC_OK;
}

/*
 * Graph Transformer attention for the selected destination rows i, every
 * head h (query at the destination, key and value at the source):
 *   e_ij = scale * sum_d Q[i,h,d] K[j,h,d]
 *   out_i[h,:] = sum_j softmax_j(e_ij) V[j,h,:],  lse[i,h] = ln sum_j exp(e_ij)
 * Q, K, V are [N, heads*D] row-major.
 */
int orc_gt(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
           const void *Q, const void *K, const void *V, int dtype, int32_t heads,
           int32_t D, double scale, const int32_t *rows, int32_t n_sel,
           double *out, double *lse, double *alpha) {
    (void)n_rows;
    int32_t HD = heads * D;
    int64_t max_deg = 0;
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        int64_t d = rowptr[i + 1] - rowptr[i];
        if (d > max_deg) max_deg = d;
    }
    double *e = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double *al = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    if (!e || !al) { free(e); free(al); return ORC_ERR; }
    int64_t alpha_pos = 0;
    for (int32_t s = 0; s < n_sel; ++s) {
        int32_t i = sel_row(rows, s);
        int64_t b = rowptr[i], deg = rowptr[i + 1] - b;
        for (int32_t h = 0; h < heads; ++h) {
            for (int64_t k = 0; k < deg; ++k) {
                int32_t j = colidx[b + k];
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    acc += widen(Q, dtype, (int64_t)i * HD + h * D + d) *
                           widen(K, dtype, (int64_t)j * HD + h * D + d);
                e[k] = scale * acc;
            }
            double L = softmax_row(e, deg, al);
            lse[(int64_t)s * heads + h] = L;
            for (int32_t d = 0; d < D; ++d) {
                double o = 0.0;
                for (int64_t k = 0; k < deg; ++k)
                    o += al[k] * widen(V, dtype, (int64_t)colidx[b + k] * HD + h * D + d);
                out[(int64_t)s * HD + h * D + d] = o;
            }
            if (alpha)
                for (int64_t k = 0; k < deg; ++k) alpha[(alpha_pos + k) * heads + h] = al[k];
        }
        alpha_pos += deg;
    }
    free(e); free(al);
    return ORC_OK;
}

/*
 * Backward of the Graph Transformer attention (IO-aware GNN layers,
 * Appendix D.2, the GT backward: Delta = <O, dO> per destination and head,
 * then the score gradient from the recomputed weights).  For row i, head h,
 * with s_ij = scale <q_i, k_j> over j in N(i), alpha = softmax_j(s), O_i =
 * sum_j alpha_ij v_j and Delta_i = <O_i, dO_i>:
 *   ds_ij  = alpha_ij (<dO_i, v_j> - Delta_i)
 *   dQ_i  += scale ds_ij k_j,  dK_j += scale ds_ij q_i,  dV_j += alpha_ij dO_i.
 * Q, K, V [n, heads*D] (dtype as orc_gt); dO, dQ, dK, dV fp64 [n, heads*D];
 * the graph is square.  dQ, dK, dV are overwritten.
 */
int orc_gt_backward(int32_t n, const int32_t *rowptr, const int32_t *colidx, const void *Q,
                    const void *K, const void *V, int dtype, int32_t heads, int32_t D, double scale,
                    const double *dO, double *dQ, double *dK, double *dV) {
    int32_t HD = heads * D;
    for (int64_t k = 0; k < (int64_t)n * HD; ++k) dQ[k] = dK[k] = dV[k] = 0.0;
    int64_t max_deg = 0;
    for (int32_t i = 0; i < n; ++i)
        if (rowptr[i + 1] - rowptr[i] > max_deg) max_deg = rowptr[i + 1] - rowptr[i];
    double *e = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double *al = malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double *o = malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
    if (!e || !al || !o) { free(e); free(al); free(o); return ORC_ERR; }
    for (int32_t i = 0; i < n; ++i) {
        int64_t b = rowptr[i], deg = rowptr[i + 1] - b;
        if (deg == 0) continue;
        for (int32_t h = 0; h < heads; ++h) {
            int64_t qo = (int64_t)i * HD + h * D;
            for (int64_t k = 0; k < deg; ++k) {
                int64_t ko = (int64_t)colidx[b + k] * HD + h * D;
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d) acc += widen(Q, dtype, qo + d) * widen(K, dtype, ko + d);
                e[k] = scale * acc;
            }
            softmax_row(e, deg, al);
            double delta = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                o[d] = 0.0;
                for (int64_t k = 0; k < deg; ++k)
                    o[d] += al[k] * widen(V, dtype, (int64_t)colidx[b + k] * HD + h * D + d);
                delta += o[d] * dO[qo + d];
            }
            for (int64_t k = 0; k < deg; ++k) {
                int64_t ko = (int64_t)colidx[b + k] * HD + h * D;
                double da = 0.0;
                for (int32_t d = 0; d < D; ++d) da += dO[qo + d] * widen(V, dtype, ko + d);
                double ds = al[k] * (da - delta);
                for (int32_t d = 0; d < D; ++d) {
                    dQ[qo + d] += scale * ds * widen(K, dtype, ko + d);
                    dK[ko + d] += scale * ds * widen(Q, dtype, qo + d);
                    dV[ko + d] += al[k] * dO[qo + d];
                }
            }
        }
    }
    free(e); free(al); free(o);
    return ORC_OK;
}

/*
 * Backward of the GATv2 attention with respect to its per-node features and
 * the attention vector (IO-aware GNN layers, Appendix D.2, the GATv2
 * backward: the weights are recomputed from the logits, the statistic
 * G_i,h = sum_j alpha_ij <dO_i, r_j> is formed per destination and head, the
 * left-feature and attention-vector gradients come from the destination
 * rows and the right-feature gradient gathers over the incoming edges of
 * each source).  For row i, head h, edge j in N(i), with x_ij = l_i + r_j
 * (the head's D channels), sigma = LeakyReLU_slope, e_ij = <a_h, sigma(x_ij)>
 * and alpha = softmax_j(e):
 *   de_ij = alpha_ij (<dO_i, r_j> - G_i)
 *   dl_i += de_ij a_h . sigma'(x_ij)
 *   dr_j += alpha_ij dO_i + de_ij a_h . sigma'(x_ij)
 *   da_h += de_ij sigma(x_ij)
 * sigma'(x) = 1 for x > 0, else slope.  Cl, Cr [n, heads*D] (dtype as
 * orc_gt; Cl == Cr for a shared projection); dO, dl, dr fp64 [n, heads*D];
 * da fp64 [heads*D].  The graph is square.  Outputs are overwritten.
 */
int orc_gatv2_backward(int32_t n, const int32_t *rowptr, const int32_t *colidx, const void *Cl,
                       const void *Cr, int dtype, const float *a, int32_t heads, int32_t D,
                       double slope, const double *dO, double *dl, double *dr, double *da) {
    int32_t HD = heads * D;
    for (int64_t k = 0; k < (int64_t)n * HD; ++k) dl[k] = dr[k] = 0.0;
    for (int32_t c = 0; c < HD; ++c) da[c] = 0.0;
    int64_t max_deg = 0;
    for (int32_t i = 0; i < n; ++i)
        if (rowptr[i + 1] - rowptr[i] > max_deg) max_deg = rowptr[i + 1] - rowptr[i];
    size_t md = (size_t)(max_deg > 0 ? max_deg : 1);
    double *e = malloc(sizeof(double) * md);
    double *al = malloc(sizeof(double) * md);
    double *p = malloc(sizeof(double) * md);
    if (!e || !al || !p) { free(e); free(al); free(p); return ORC_ERR; }
    for (int32_t i = 0; i < n; ++i) {
        int64_t b = rowptr[i], deg = rowptr[i + 1] - b;
        if (deg == 0) continue;
        for (int32_t h = 0; h < heads; ++h) {
            int64_t io = (int64_t)i * HD + h * D;
            /* logits, weights and <dO_i, r_j> */
            for (int64_t k = 0; k < deg; ++k) {
                int64_t jo = (int64_t)colidx[b + k] * HD + h * D;
                double acc = 0.0, pr = 0.0;
                for (int32_t d = 0; d < D; ++d) {
                    double x = widen(Cl, dtype, io + d) + widen(Cr, dtype, jo + d);
                    acc += (double)a[h * D + d] * (x > 0.0 ? x : slope * x);
                    pr += dO[io + d] * widen(Cr, dtype, jo + d);
                }
                e[k] = acc;
                p[k] = pr;
            }
            softmax_row(e, deg, al);
            double G = 0.0;
            for (int64_t k = 0; k < deg; ++k) G += al[k] * p[k];
            for (int64_t k = 0; k < deg; ++k) {
                int64_t jo = (int64_t)colidx[b + k] * HD + h * D;
                double de = al[k] * (p[k] - G);
                for (int32_t d = 0; d < D; ++d) {
                    double x = widen(Cl, dtype, io + d) + widen(Cr, dtype, jo + d);
                    double g = de * (double)a[h * D + d] * (x > 0.0 ? 1.0 : slope);
                    dl[io + d] += g;
                    dr[jo + d] += al[k] * dO[io + d] + g;
                    da[h * D + d] += de * (x > 0.0 ? x : slope * x);
                }
            }
        }
    }
    free(e); free(al); free(p);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* block-sparse tiles (IO-aware GNN layers, Appendix D.3, WSB format)  */
/* ------------------------------------------------------------------ */

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

typedef struct { int64_t cnt; int32_t id; int32_t k; } orc_colcount;

/* descending count, then ascending column id */
static int cmp_colcount(const void *a, const void *b) {
    const orc_colcount *x = a, *y = b;
    if (x->cnt != y->cnt) return x->cnt > y->cnt ? -1 : 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* index of column j in the sorted unique list U[0..nu) (j is present) */
static int64_t find_col(const int32_t *U, int64_t nu, int32_t j) {
    int64_t lo = 0, hi = nu - 1;
    while (lo < hi) {
        int64_t mid = (lo + hi) / 2;
        if (U[mid] < j) lo = mid + 1; else hi = mid;
    }
    return lo;
}

/*
 * Rows are cut into windows of 16 and groups of 8 windows (128 rows).  For a
 * group g, U_g = the sorted unique source columns of its rows; column block
 * b holds U_g[16b .. 16b+16) (missing entries padded with column 0 and never
 * masked in).  The tile (window w, block b) is 16x16 with a 256-bit mask,
 * bit r*16+c set iff the edge U_g[16b+c] -> 16w+r exists (word (r*16+c)/64,
 * bit (r*16+c)%64).  A tile is kept iff its popcount p >= 1 and
 * (float)p / 256.0f >= threshold (fp32 comparison).  A block is listed iff at
 * least one of its 8 tiles is kept; listed blocks keep ascending b.  Masks of
 * tiles that are not kept are stored as zero.  Edges of tiles that are not
 * kept form the residual CSR (same rows, ascending columns).
 *
 * counts[0..3] = {n_blocks, n_tiles_kept, nnz_tiles, nnz_residual}.
 * Output arrays may be NULL (count only).  grp_blk_offset [n_groups+1],
 * blk_cols [n_blocks*16], blk_mask [n_blocks*8*4], res_rowptr [n_rows+1],
 * res_colidx [nnz_residual].
 *
 * packing 0 orders U_g by ascending column id, the plain reading of the
 * pages' "sorted" columns.  packing 1 orders it by descending count of the
 * column's edges into the group's rows, ties by ascending id, so the
 * columns that carry most edges share the first blocks and their tiles
 * fill up (the fill-raising packing the threshold rule benefits from); the
 * set of columns, and so the number of blocks at threshold 0, is the same.
 */
int orc_blocksparse_packed(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
                           float threshold, int packing, int64_t *counts,
                           int32_t *grp_blk_offset, int32_t *blk_cols, uint64_t *blk_mask,
                           int32_t *res_rowptr, int32_t *res_colidx) {
    int32_t n_groups = (n_rows + 127) / 128;
    int64_t n_blocks = 0, n_kept = 0, nnz_tiles = 0, nnz_res = 0;
    int64_t max_ge = 0;
    for (int32_t g = 0; g < n_groups; ++g) {
        int32_t r0 = g * 128, r1 = r0 + 128 < n_rows ? r0 + 128 : n_rows;
        int64_t ge = rowptr[r1] - rowptr[r0];
        if (ge > max_ge) max_ge = ge;
    }
    size_t mg = (size_t)(max_ge > 0 ? max_ge : 1);
    int32_t *U = malloc(sizeof(int32_t) * mg);
    int32_t *P = malloc(sizeof(int32_t) * mg);      /* packed order of U */
    int64_t *rank = malloc(sizeof(int64_t) * mg);   /* position in P of U[k] */
    orc_colcount *cc = malloc(sizeof(orc_colcount) * mg);
    /* per group: masks[block][window][4] */
    int64_t max_blocks = (max_ge + 15) / 16;
    uint64_t *masks = malloc(sizeof(uint64_t) * (size_t)(max_blocks > 0 ? max_blocks : 1) * 32);
    uint8_t *kept = malloc((size_t)(max_blocks > 0 ? max_blocks : 1) * 8);
    if (!U || !P || !rank || !cc || !masks || !kept) {
        free(U); free(P); free(rank); free(cc); free(masks); free(kept);
        return ORC_ERR;
    }
    if (res_rowptr) res_rowptr[0] = 0;
    if (grp_blk_offset) grp_blk_offset[0] = 0;
    for (int32_t g = 0; g < n_groups; ++g) {
        int32_t r0 = g * 128, r1 = r0 + 128 < n_rows ? r0 + 128 : n_rows;
        int64_t ge = rowptr[r1] - rowptr[r0];
        memcpy(U, colidx + rowptr[r0], sizeof(int32_t) * (size_t)ge);
        qsort(U, (size_t)ge, sizeof(int32_t), cmp_i32);
        int64_t nu = 0;
        for (int64_t k = 0; k < ge; ++k)
            if (nu == 0 || U[nu - 1] != U[k]) U[nu++] = U[k];
        /* the packed order P of the columns and the position of each */
        for (int64_t k = 0; k < nu; ++k) { cc[k].cnt = 0; cc[k].id = U[k]; cc[k].k = (int32_t)k; }
        if (packing == 1) {
            for (int64_t e = rowptr[r0]; e < rowptr[r1]; ++e) cc[find_col(U, nu, colidx[e])].cnt++;
            qsort(cc, (size_t)nu, sizeof(orc_colcount), cmp_colcount);
        }
        for (int64_t q = 0; q < nu; ++q) { P[q] = cc[q].id; rank[cc[q].k] = q; }
        int64_t nb = (nu + 15) / 16;
        memset(masks, 0, sizeof(uint64_t) * (size_t)nb * 32);
        /* place every edge of the group */
        for (int32_t i = r0; i < r1; ++i) {
            int32_t w = (i - r0) / 16, r = (i - r0) % 16;
            for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
                int64_t lo = rank[find_col(U, nu, colidx[e])];
                int64_t b = lo / 16, c = lo % 16, bit = r * 16 + c;
                masks[(b * 8 + w) * 4 + bit / 64] |= 1ull << (bit % 64);
            }
        }
        for (int64_t b = 0; b < nb; ++b) {
            int any = 0;
            for (int32_t w = 0; w < 8; ++w) {
                int p = 0;
                for (int q = 0; q < 4; ++q) p += __builtin_popcountll(masks[(b * 8 + w) * 4 + q]);
                int k = (p >= 1) && ((float)p / 256.0f >= threshold);
                kept[b * 8 + w] = (uint8_t)k;
                if (k) { any = 1; n_kept++; nnz_tiles += p; }
            }
            if (any) {
                if (blk_cols)
                    for (int c = 0; c < 16; ++c)
                        blk_cols[n_blocks * 16 + c] = (16 * b + c < nu) ? P[16 * b + c] : 0;
                if (blk_mask)
                    for (int32_t w = 0; w < 8; ++w)
                        for (int q = 0; q < 4; ++q)
                            blk_mask[(n_blocks * 8 + w) * 4 + q] =
                                kept[b * 8 + w] ? masks[(b * 8 + w) * 4 + q] : 0;
                n_blocks++;
            }
        }
        if (grp_blk_offset) grp_blk_offset[g + 1] = (int32_t)n_blocks;
        /* residual edges, in row order then ascending column */
        for (int32_t i = r0; i < r1; ++i) {
            int32_t w = (i - r0) / 16;
            for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
                int32_t j = colidx[e];
                int64_t lo = rank[find_col(U, nu, j)];
                if (!kept[(lo / 16) * 8 + w]) {
                    if (res_colidx) res_colidx[nnz_res] = j;
                    nnz_res++;
                }
            }
            if (res_rowptr) res_rowptr[i + 1] = (int32_t)nnz_res;
        }
    }
    counts[0] = n_blocks;
    counts[1] = n_kept;
    counts[2] = nnz_tiles;
    counts[3] = nnz_res;
    free(U); free(P); free(rank); free(cc); free(masks); free(kept);
    return ORC_OK;
}

/* The layout with columns in ascending id order (packing 0). */
int orc_blocksparse(int32_t n_rows, const int32_t *rowptr, const int32_t *colidx,
                    float threshold, int64_t *counts, int32_t *grp_blk_offset,
                    int32_t *blk_cols, uint64_t *blk_mask, int32_t *res_rowptr,
                    int32_t *res_colidx) {
    return orc_blocksparse_packed(n_rows, rowptr, colidx, threshold, 0, counts, grp_blk_offset,
                                  blk_cols, blk_mask, res_rowptr, res_colidx);
}

/* ------------------------------------------------------------------ */
/* vertex orderings                                                    */
/* ------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea, Flood 2014): one step of the generator started
 * from state x. */
uint64_t orc_splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

typedef struct { uint64_t k; int32_t id; } key_id;

static int cmp_key_id(const void *a, const void *b) {
    const key_id *x = a, *y = b;
    if (x->k != y->k) return x->k < y->k ? -1 : 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* perm[new] = old.  Random order: ascending (splitmix64(seed ^ id), id). */
int orc_perm_random(int32_t n, uint64_t seed, int32_t *perm) {
    key_id *v = malloc(sizeof(key_id) * (size_t)(n > 0 ? n : 1));
    if (!v) return ORC_ERR;
    for (int32_t i = 0; i < n; ++i) { v[i].k = orc_splitmix64(seed ^ (uint64_t)i); v[i].id = i; }
    qsort(v, (size_t)n, sizeof(key_id), cmp_key_id);
    for (int32_t i = 0; i < n; ++i) perm[i] = v[i].id;
    free(v);
    return ORC_OK;
}

/* Degree order: descending total degree d_in + d_out (as stored, self-loops
 * included), ties by ascending id. */
int orc_perm_degree(int32_t n, const int32_t *rowptr, const int32_t *colidx,
                    int32_t *perm) {
    int64_t *deg = calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    key_id *v = malloc(sizeof(key_id) * (size_t)(n > 0 ? n : 1));
    if (!deg || !v) { free(deg); free(v); return ORC_ERR; }
    for (int32_t i = 0; i < n; ++i) deg[i] += rowptr[i + 1] - rowptr[i];
    for (int64_t e = 0; e < rowptr[n]; ++e) deg[colidx[e]]++;
    for (int32_t i = 0; i < n; ++i) { v[i].k = (uint64_t)(INT64_MAX - deg[i]); v[i].id = i; }
    qsort(v, (size_t)n, sizeof(key_id), cmp_key_id);
    for (int32_t i = 0; i < n; ++i) perm[i] = v[i].id;
    free(deg); free(v);
    return ORC_OK;
}

/* symmetric adjacency S = (A + A^T) without self-loops, deduplicated */
static int symmetrize(int32_t n, const int32_t *rowptr, const int32_t *colidx,
                      int64_t **sp_out, int32_t **sc_out) {
    int64_t m = rowptr[n];
    int64_t *cnt = calloc((size_t)n + 1, sizeof(int64_t));
    if (!cnt) return ORC_ERR;
    for (int32_t i = 0; i < n; ++i)
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e)
            if (colidx[e] != i) { cnt[i + 1]++; cnt[colidx[e] + 1]++; }
    for (int32_t i = 0; i < n; ++i) cnt[i + 1] += cnt[i];
    int32_t *adj = malloc(sizeof(int32_t) * (size_t)(cnt[n] > 0 ? cnt[n] : 1));
    int64_t *pos = malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!adj || !pos) { free(cnt); free(adj); free(pos); return ORC_ERR; }
    (void)m;
    for (int32_t i = 0; i < n; ++i) pos[i] = cnt[i];
    for (int32_t i = 0; i < n; ++i)
        for (int64_t e = rowptr[i]; e < rowptr[i + 1]; ++e) {
            int32_t j = colidx[e];
            if (j == i) continue;
            adj[pos[i]++] = j;
            adj[pos[j]++] = i;
        }
    /* sort + dedupe each list, compacting */
    int64_t w = 0;
    int64_t prev_start = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t b = cnt[i], e = cnt[i + 1];
        qsort(adj + b, (size_t)(e - b), sizeof(int32_t), cmp_i32);
        int64_t start = w;
        for (int64_t k = b; k < e; ++k)
            if (w == start || adj[w - 1] != adj[k]) adj[w++] = adj[k];
        cnt[i] = prev_start;
        prev_start = w;
        (void)start;
    }
    cnt[n] = w;
    /* cnt[i] now holds the compacted start of list i */
    free(pos);
    *sp_out = cnt;
    *sc_out = adj;
    return ORC_OK;
}

static int32_t *g_sdeg; /* degree table used by the comparators below */

static int cmp_deg_id(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    if (g_sdeg[x] != g_sdeg[y]) return g_sdeg[x] < g_sdeg[y] ? -1 : 1;
    return (x > y) - (x < y);
}

/*
 * Reverse Cuthill-McKee on S = A + A^T (self-loops dropped).  Each connected
 * component starts at the unvisited node of smallest degree (lowest id on
 * ties); breadth-first, each dequeued node appends its unvisited neighbours
 * in ascending (degree, id) order; the final sequence is reversed.
 * perm[new] = old.
 */
int orc_perm_rcm(int32_t n, const int32_t *rowptr, const int32_t *colidx,
                 int32_t *perm) {
    int64_t *sp;
    int32_t *sc;
    if (symmetrize(n, rowptr, colidx, &sp, &sc) != ORC_OK) return ORC_ERR;
    int32_t *deg = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t *by_deg = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t *order = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t *tmp = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    uint8_t *vis = calloc((size_t)(n > 0 ? n : 1), 1);
    if (!deg || !by_deg || !order || !tmp || !vis) {
        free(sp); free(sc); free(deg); free(by_deg); free(order); free(tmp); free(vis);
        return ORC_ERR;
    }
    for (int32_t i = 0; i < n; ++i) { deg[i] = (int32_t)(sp[i + 1] - sp[i]); by_deg[i] = i; }
    g_sdeg = deg;
    qsort(by_deg, (size_t)n, sizeof(int32_t), cmp_deg_id);
    int32_t len = 0, scan = 0;
    while (len < n) {
        while (vis[by_deg[scan]]) ++scan;
        int32_t start = by_deg[scan];
        vis[start] = 1;
        order[len++] = start;
        for (int32_t head = len - 1; head < len; ++head) {
            int32_t u = order[head];
            int32_t t = 0;
            for (int64_t k = sp[u]; k < sp[u + 1]; ++k)
                if (!vis[sc[k]]) { vis[sc[k]] = 1; tmp[t++] = sc[k]; }
            qsort(tmp, (size_t)t, sizeof(int32_t), cmp_deg_id);
            for (int32_t k = 0; k < t; ++k) order[len++] = tmp[k];
        }
    }
    for (int32_t k = 0; k < n; ++k) perm[k] = order[n - 1 - k];
    free(sp); free(sc); free(deg); free(by_deg); free(order); free(tmp); free(vis);
    return ORC_OK;
}

/*
 * Relabel a square CSR by perm (perm[new] = old, inv[old] = new): new row r
 * is old row perm[r] with every column c replaced by inv[c], columns
 * re-sorted ascending.  Feature rows follow as X_new[r] = X[perm[r]].
 */
int orc_apply_perm(int32_t n, const int32_t *rowptr, const int32_t *colidx,
                   const int32_t *perm, int32_t *rowptr_out, int32_t *colidx_out) {
    int32_t *inv = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    if (!inv) return ORC_ERR;
    for (int32_t k = 0; k < n; ++k) inv[perm[k]] = k;
    rowptr_out[0] = 0;
    for (int32_t r = 0; r < n; ++r) {
        int32_t o = perm[r];
        int32_t b = rowptr_out[r];
        int32_t d = rowptr[o + 1] - rowptr[o];
        for (int32_t k = 0; k < d; ++k) colidx_out[b + k] = inv[colidx[rowptr[o] + k]];
        qsort(colidx_out + b, (size_t)d, sizeof(int32_t), cmp_i32);
        rowptr_out[r + 1] = b + d;
    }
    free(inv);
    return ORC_OK;
}
