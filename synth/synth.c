/*
 * Seeded synthetic inputs: graphs in CSR form (rows = destinations, columns =
 * sources, ascending within each row, duplicates removed, exactly one
 * self-loop per node) and dense node features.
 *
 * This module holds no arithmetic of the aggregation method itself; it only
 * draws random numbers and lays out the CSR input format.  It serves both the
 * CUDA library's tests/benchmarks and the CPU oracle's tests.
 *
 * Random numbers: a counter-based generator, SplitMix64 (Steele, Lea, Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), evaluated at
 * key(seed, stream) + index, so every draw is a pure function of
 * (seed, stream, index) and parallel loops reproduce the serial stream.
 * Uniform doubles take the top 53 bits; normals use Box-Muller.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return sm64(sm64(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

static inline uint64_t draw(uint64_t key, uint64_t index) {
    return sm64(key + index * 0x9E3779B97F4A7C15ull);
}

static inline double unit(uint64_t u) { /* [0,1) */
    return (double)(u >> 11) * (1.0 / 9007199254740992.0);
}

/* uniform integer in [0, n) by 64x64->128 multiply-shift */
static inline uint64_t below(uint64_t u, uint64_t n) {
    return (uint64_t)(((unsigned __int128)u * n) >> 64);
}

uint64_t synth_splitmix64(uint64_t x) { return sm64(x); }

/* ------------------------------------------------------------------ */
/* features                                                            */
/* ------------------------------------------------------------------ */

void synth_uniform_f32(float *out, int64_t n, double lo, double hi,
                       uint64_t seed, uint64_t stream) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(lo + (hi - lo) * unit(draw(key, (uint64_t)i)));
}

static void normal_fill(double *tmp_or_null, float *out_f32, uint16_t *out_bf16,
                        int64_t n, double mean, double std, uint64_t seed,
                        uint64_t stream) {
    (void)tmp_or_null;
    uint64_t key = stream_key(seed, stream);
    int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < pairs; ++p) {
        double u1 = 1.0 - unit(draw(key, 2 * (uint64_t)p));     /* (0,1] */
        double u2 = unit(draw(key, 2 * (uint64_t)p + 1));
        double r = sqrt(-2.0 * log(u1));
        double t = 6.283185307179586 * u2;
        double z[2] = {r * cos(t), r * sin(t)};
        for (int k = 0; k < 2; ++k) {
            int64_t i = 2 * p + k;
            if (i >= n) break;
            float f = (float)(mean + std * z[k]);
            if (out_f32) out_f32[i] = f;
            if (out_bf16) {
                uint32_t b;
                memcpy(&b, &f, 4);
                /* fp32 -> bf16, round to nearest even on the bit pattern
                 * (inputs are finite) */
                uint32_t lsb = (b >> 16) & 1u;
                b += 0x7FFFu + lsb;
                out_bf16[i] = (uint16_t)(b >> 16);
            }
        }
    }
}

void synth_normal_f32(float *out, int64_t n, double mean, double std,
                      uint64_t seed, uint64_t stream) {
    normal_fill(NULL, out, NULL, n, mean, std, seed, stream);
}

void synth_normal_bf16(uint16_t *out, int64_t n, double mean, double std,
                       uint64_t seed, uint64_t stream) {
    normal_fill(NULL, NULL, out, n, mean, std, seed, stream);
}

/* ------------------------------------------------------------------ */
/* CSR assembly from a (dst, src) edge list                             */
/* ------------------------------------------------------------------ */

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

static void sort_small(int32_t *v, int64_t n) {
    if (n > 32) { qsort(v, (size_t)n, sizeof(int32_t), cmp_i32); return; }
    for (int64_t i = 1; i < n; ++i) {
        int32_t x = v[i];
        int64_t j = i - 1;
        while (j >= 0 && v[j] > x) { v[j + 1] = v[j]; --j; }
        v[j + 1] = x;
    }
}

/*
 * Build CSR by destination from parallel arrays dst[], src[] of length m.
 * Self-loops in the list are dropped, duplicates removed, and one self-loop
 * per node added.  rowptr must hold n+1 entries; *colidx_out is malloc'ed and
 * owned by the caller (free with synth_free).  Returns nnz, or -1 on OOM.
 */
static int64_t assemble(int32_t n, const int32_t *dst, const int32_t *src,
                        int64_t m, int32_t *rowptr, int32_t **colidx_out) {
    int64_t *cnt = calloc((size_t)n + 1, sizeof(int64_t));
    if (!cnt) return -1;
    for (int64_t e = 0; e < m; ++e)
        if (dst[e] != src[e]) cnt[dst[e] + 1]++;
    for (int32_t i = 0; i < n; ++i) cnt[i + 1] += cnt[i] + 0;
    /* +1 slot per row for the self-loop */
    int64_t total = cnt[n] + n;
    int32_t *tmp = malloc((size_t)total * sizeof(int32_t));
    int64_t *pos = malloc((size_t)n * sizeof(int64_t));
    if (!tmp || !pos) { free(cnt); free(tmp); free(pos); return -1; }
    for (int32_t i = 0; i < n; ++i) pos[i] = cnt[i] + i;
    for (int64_t e = 0; e < m; ++e)
        if (dst[e] != src[e]) tmp[pos[dst[e]]++] = src[e];
    for (int32_t i = 0; i < n; ++i) tmp[pos[i]++] = i; /* self-loop */
    /* sort + dedupe each row in place, compacting */
    int64_t w = 0;
    rowptr[0] = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t b = cnt[i] + i, e = cnt[i + 1] + i + 1;
        sort_small(tmp + b, e - b);
        int64_t row_start = w;
        for (int64_t k = b; k < e; ++k)
            if (w == row_start || tmp[w - 1] != tmp[k]) tmp[w++] = tmp[k];
        rowptr[i + 1] = (int32_t)w;
    }
    free(cnt);
    free(pos);
    int32_t *col = realloc(tmp, (size_t)(w > 0 ? w : 1) * sizeof(int32_t));
    *colidx_out = col ? col : tmp;
    return w;
}

void synth_free(void *p) { free(p); }

/* Copy a malloc'ed colidx into a caller buffer and free it. */
void synth_take(int32_t *dst, int32_t *src, int64_t nnz) {
    memcpy(dst, src, (size_t)nnz * sizeof(int32_t));
    free(src);
}

/*
 * Erdos-Renyi G(n, m): m distinct ordered pairs (src -> dst), src != dst,
 * drawn uniformly with rejection (draw order fixed by the stream index).
 */
int64_t synth_er(int32_t n, int64_t m, uint64_t seed, int32_t *rowptr,
                 int32_t **colidx_out) {
    uint64_t key = stream_key(seed, 100);
    uint64_t nn = (uint64_t)n * (uint64_t)n;
    uint8_t *seen = calloc((size_t)((nn + 7) / 8), 1);
    int32_t *dst = malloc((size_t)m * sizeof(int32_t));
    int32_t *src = malloc((size_t)m * sizeof(int32_t));
    if (!seen || !dst || !src) { free(seen); free(dst); free(src); return -1; }
    int64_t got = 0;
    uint64_t idx = 0;
    while (got < m) {
        uint64_t s = below(draw(key, idx++), (uint64_t)n);
        uint64_t d = below(draw(key, idx++), (uint64_t)n);
        if (s == d) continue;
        uint64_t bit = d * (uint64_t)n + s;
        if (seen[bit >> 3] & (1u << (bit & 7))) continue;
        seen[bit >> 3] |= (uint8_t)(1u << (bit & 7));
        dst[got] = (int32_t)d;
        src[got] = (int32_t)s;
        ++got;
    }
    int64_t nnz = assemble(n, dst, src, m, rowptr, colidx_out);
    free(seen); free(dst); free(src);
    return nnz;
}

/*
 * R-MAT (Chakrabarti, Zhan, Faloutsos 2004): ef * 2^scale edges; for each edge
 * and each of `scale` bit levels one uniform draw picks a quadrant:
 *   u < a          : (src bit 0, dst bit 0)
 *   u < a+b        : (src bit 0, dst bit 1)
 *   u < a+b+c      : (src bit 1, dst bit 0)
 *   otherwise      : (src bit 1, dst bit 1)
 * Level k sets bit k (LSB first).  No noise, no label scrambling.
 */
int64_t synth_rmat(int32_t scale, int32_t edge_factor, double a, double b,
                   double c, uint64_t seed, int32_t *rowptr,
                   int32_t **colidx_out) {
    int32_t n = (int32_t)1 << scale;
    int64_t m = (int64_t)edge_factor * n;
    uint64_t key = stream_key(seed, 200);
    int32_t *dst = malloc((size_t)m * sizeof(int32_t));
    int32_t *src = malloc((size_t)m * sizeof(int32_t));
    if (!dst || !src) { free(dst); free(src); return -1; }
    double ab = a + b, abc = a + b + c;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < m; ++e) {
        uint32_t s = 0, d = 0;
        for (int32_t k = 0; k < scale; ++k) {
            double u = unit(draw(key, (uint64_t)e * (uint64_t)scale + (uint64_t)k));
            if (u < a) {
            } else if (u < ab) {
                d |= 1u << k;
            } else if (u < abc) {
                s |= 1u << k;
            } else {
                s |= 1u << k;
                d |= 1u << k;
            }
        }
        dst[e] = (int32_t)d;
        src[e] = (int32_t)s;
    }
    int64_t nnz = assemble(n, dst, src, m, rowptr, colidx_out);
    free(dst); free(src);
    return nnz;
}

/*
 * Locally dense clustered graph: node ids [cs*k, cs*k+cs) form cluster k.
 * Every ordered pair (src -> dst), src != dst, inside a cluster is an edge
 * with probability p; each such edge then, with probability rewire, has its
 * source replaced by a node drawn uniformly from outside the cluster
 * (destination kept).  Duplicates removed, one self-loop per node added.
 */
int64_t synth_clustered(int32_t n_clusters, int32_t cluster_size, double p,
                        double rewire, uint64_t seed, int32_t *rowptr,
                        int32_t **colidx_out) {
    int64_t n64 = (int64_t)n_clusters * cluster_size;
    int32_t n = (int32_t)n64;
    uint64_t key = stream_key(seed, 300);
    int64_t pairs = (int64_t)cluster_size * (cluster_size - 1);
    int64_t cap = (int64_t)((double)n_clusters * (double)pairs * p * 1.05) + 1024;
    int32_t *dst = malloc((size_t)cap * sizeof(int32_t));
    int32_t *src = malloc((size_t)cap * sizeof(int32_t));
    if (!dst || !src) { free(dst); free(src); return -1; }
    int64_t m = 0;
    for (int32_t k = 0; k < n_clusters; ++k) {
        int64_t base = (int64_t)k * cluster_size;
        for (int32_t di = 0; di < cluster_size; ++di) {
            for (int32_t si = 0; si < cluster_size; ++si) {
                if (si == di) continue;
                uint64_t idx = (uint64_t)((base + di) * cluster_size + si) * 3u;
                if (unit(draw(key, idx)) >= p) continue;
                int64_t s = base + si;
                if (unit(draw(key, idx + 1)) < rewire) {
                    uint64_t o = below(draw(key, idx + 2), (uint64_t)(n64 - cluster_size));
                    s = (int64_t)o < base ? (int64_t)o : (int64_t)o + cluster_size;
                }
                if (m == cap) { free(dst); free(src); return -1; }
                dst[m] = (int32_t)(base + di);
                src[m] = (int32_t)s;
                ++m;
            }
        }
    }
    int64_t nnz = assemble(n, dst, src, m, rowptr, colidx_out);
    free(dst); free(src);
    return nnz;
}

int synth_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
