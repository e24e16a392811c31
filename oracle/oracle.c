/*
 * oracle.c -- plain, slow CPU oracle of the DLRM sparse forward and of its
 * training step (interaction backward, per-row gradient reduction, row-wise
 * Adagrad).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA library, and neither side imports the other.
 *
 * Every function is the plain definition written out as loops, accumulated in
 * double precision and rounded once to float at the end.  The only liberty
 * taken is an OpenMP loop over independent samples (or tables), which changes
 * no arithmetic.
 *
 * Sources (web pages, cited by title and section):
 *   [robocikowo]  "DLRM" (robocikowo.com), paragraph "Forward pass ... cztery
 *                 etapy", steps (2) embedding lookup of width D, (3) N x N
 *                 pairwise dot products, strict upper triangle of N(N-1)/2
 *                 values, (4) concatenation with the bottom-MLP output;
 *                 training with SGD/Adagrad.  Also its embedding-table
 *                 paragraph (E_i : V_i x D) and interaction-layer paragraph
 *                 (N vectors = bottom-MLP output + N-1 embeddings).
 *   [glossary]    "Deep Learning Recommendation Model (DLRM)"
 *                 (notes.helloworld.co.in), section "The architecture":
 *                 vectors of equal width, explicit pairwise dot products,
 *                 concatenated with the dense output.
 *   [vinsonli]    "The embedding table is the model": multi-valued sparse
 *                 features (several IDs per feature -> a bag of rows); dot
 *                 products of every pair, concatenated with the dense vector.
 *   [technolynx]  "DLRM explained", section "How does DLRM actually work?":
 *                 one lookup per feature, each returning a learned vector.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - bags: CSR, table-major: bag (t,b) holds indices[offsets[t*B+b] ..
 *     offsets[t*B+b+1]); indices are rows local to table t;
 *   - pooling: sum or mean; an empty bag pools to zeros; duplicates count;
 *     a sum starts from its first term (so a single -0.0 stays -0.0);
 *   - an out-of-range index contributes nothing but still counts in L;
 *     a bag whose range is negative, reversed or past nnz is treated as
 *     empty; both raise a flag in the returned status;
 *   - output row = [x (D values, copied), z(i,j) for i<j in row-major order];
 *     vector 0 is x, vectors 1..T are the pooled bags in table order;
 *   - Adagrad is row-wise: one accumulator per row, A += mean_d(g_d^2), then
 *     w_d -= lr * g_d / (sqrt(A) + eps); the gradients of all lookups of a row
 *     in one step are summed first (one update per touched row); rows not
 *     touched are left alone.
 *   - plain SGD (the other rule the same sentence names) is w_d -= lr * g_d on
 *     the same per-row gradient sums: no momentum, no weight decay;
 *   - the hashing of raw feature IDs into a table of V_t rows ("Deep Learning
 *     Recommendation Model (DLRM)", notes.helloworld.co.in, "Why it is mostly
 *     a systems problem") is read as the plainest hash: the ID, taken as an
 *     unsigned 64-bit integer, modulo V_t.
 */
#include <math.h>
#include <omp.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_INDEX_OOB 2
#define ORACLE_BAD_OFFSETS 4

#define ORACLE_F32 0
#define ORACLE_BF16 1

#define ORACLE_SUM 0
#define ORACLE_MEAN 1

#define ORACLE_ADAGRAD 0
#define ORACLE_SGD 1

/* Threads of the OpenMP loops over independent samples or tables (n >= 1);
 * returns the count now in effect.  Changes no arithmetic: each sample's and
 * each table's loops run the same way on any number of threads. */
int oracle_set_threads(int n)
{
    if (n >= 1)
        omp_set_num_threads(n);
    return omp_get_max_threads();
}

/* One table element widened to double.  bf16 is the top half of an fp32
 * pattern, so widening is exact. */
static double table_elem(const void *table, int dtype, int64_t row, int D, int d)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)table)[row * (int64_t)D + d];
    uint32_t bits = (uint32_t)((const uint16_t *)table)[row * (int64_t)D + d] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Bag (t,b) as a half-open range of indices[]; 0 if the range is valid. */
static int bag_range(const int64_t *offsets, int64_t bag, int64_t nnz,
                     int64_t *lo, int64_t *hi)
{
    int64_t a = offsets[bag], e = offsets[bag + 1];
    if (a < 0 || e < a || e > nnz) {
        *lo = *hi = 0;
        return ORACLE_BAD_OFFSETS;
    }
    *lo = a;
    *hi = e;
    return ORACLE_OK;
}

/* Step (2) of the forward pass [robocikowo], with multi-valued features
 * pooled [vinsonli]:  P[b][t][:] = pool_{p in bag(t,b)} E_t[indices[p]][:].
 *
 * pooled      out, [B][T][D] float
 * pooled_abs  out, nullable, [B][T][D] double: the matching pool of |terms|,
 *             the scale against which a rounding error is measured.
 * Returns a bit set of ORACLE_INDEX_OOB / ORACLE_BAD_OFFSETS. */
int oracle_embbag(int T, int D, int dtype, const void *const *tables,
                  const int64_t *num_rows, int64_t B, int64_t nnz,
                  const int64_t *indices, const int64_t *offsets, int mode,
                  float *pooled, double *pooled_abs)
{
    int status = ORACLE_OK;
    if (offsets[0] != 0 || offsets[(int64_t)T * B] != nnz)
        status |= ORACLE_BAD_OFFSETS;

#pragma omp parallel for schedule(static) reduction(| : status)
    for (int64_t b = 0; b < B; ++b) {
        double *s = malloc(sizeof(double) * 2 * (size_t)D);
        double *a = s + D;
        for (int t = 0; t < T; ++t) {
            int64_t lo, hi;
            status |= bag_range(offsets, (int64_t)t * B + b, nnz, &lo, &hi);
            int64_t L = hi - lo;
            int started = 0;
            for (int d = 0; d < D; ++d)
                s[d] = a[d] = 0.0;
            for (int64_t p = lo; p < hi; ++p) {
                int64_t r = indices[p];
                if (r < 0 || r >= num_rows[t]) {
                    status |= ORACLE_INDEX_OOB;
                    continue;
                }
                for (int d = 0; d < D; ++d) {
                    double v = table_elem(tables[t], dtype, r, D, d);
                    s[d] = started ? s[d] + v : v;
                    a[d] += fabs(v);
                }
                started = 1;
            }
            float *P = pooled + ((size_t)b * T + t) * D;
            for (int d = 0; d < D; ++d) {
                double v = s[d], av = a[d];
                if (L == 0 || !started) {
                    v = 0.0;
                    av = 0.0;
                } else if (mode == ORACLE_MEAN) {
                    v /= (double)L;
                    av /= (double)L;
                }
                P[d] = (float)v;
                if (pooled_abs)
                    pooled_abs[((size_t)b * T + t) * D + d] = av;
            }
        }
        free(s);
    }
    return status;
}

/* Position of the pair (i,j), i<j, in the row-major strict upper triangle of
 * an N x N matrix. */
static int64_t tri_pos(int64_t i, int64_t j, int64_t N)
{
    return i * N - i * (i + 1) / 2 + (j - i - 1);
}

/* Vector k of sample b: 0 is the dense vector x, 1..T the pooled bags. */
static const float *vec(const float *dense, const float *pooled, int64_t b,
                        int T, int D, int k)
{
    return k == 0 ? dense + (size_t)b * D
                  : pooled + ((size_t)b * T + (k - 1)) * D;
}

/* Steps (3)-(4) of the forward pass [robocikowo]; [glossary] "The
 * architecture":  out[b] = [x_b, z_b(i,j) for 0 <= i < j < N],
 * z(i,j) = sum_d V_i[d] * V_j[d], with V = [x_b, P_b,0, ..., P_b,T-1].
 *
 * out      out, [B][D + N(N-1)/2] float
 * out_abs  out, nullable, same shape, double: |x| for the first D entries and
 *          sum_d |V_i[d] V_j[d]| for the triangle. */
void oracle_interact(int64_t B, int T, int D, const float *dense,
                     const float *pooled, float *out, double *out_abs)
{
    const int N = T + 1;
    const int64_t K = (int64_t)N * (N - 1) / 2;
    const int64_t W = D + K;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        float *o = out + (size_t)b * W;
        const float *x = dense + (size_t)b * D;
        memcpy(o, x, sizeof(float) * (size_t)D);
        if (out_abs)
            for (int d = 0; d < D; ++d)
                out_abs[(size_t)b * W + d] = fabs((double)x[d]);
        for (int i = 0; i < N; ++i) {
            const float *vi = vec(dense, pooled, b, T, D, i);
            for (int j = i + 1; j < N; ++j) {
                const float *vj = vec(dense, pooled, b, T, D, j);
                double z = 0.0, za = 0.0;
                for (int d = 0; d < D; ++d) {
                    double p = (double)vi[d] * (double)vj[d];
                    z += p;
                    za += fabs(p);
                }
                int64_t k = D + tri_pos(i, j, N);
                o[k] = (float)z;
                if (out_abs)
                    out_abs[(size_t)b * W + k] = za;
            }
        }
    }
}

/* The fused forward: pool, then interact on the pooled vectors rounded to
 * float (the rounding the forward output carries).  pooled_save, if not
 * null, receives P.  Returns the embbag status bits. */
int oracle_sparse_fwd(int T, int D, int dtype, const void *const *tables,
                      const int64_t *num_rows, int64_t B, int64_t nnz,
                      const int64_t *indices, const int64_t *offsets, int mode,
                      const float *dense, float *out, double *out_abs,
                      float *pooled_save)
{
    float *P = pooled_save ? pooled_save
                           : malloc(sizeof(float) * (size_t)B * T * D);
    int st = oracle_embbag(T, D, dtype, tables, num_rows, B, nnz, indices,
                           offsets, mode, P, NULL);
    oracle_interact(B, T, D, dense, P, out, out_abs);
    if (!pooled_save)
        free(P);
    return st;
}

/* Backward of out[b] = [x, triu(V V^T)] with respect to V, from calculus on
 * the forward definition:  with g(i,j) = g(j,i) = grad_out[b][D + pos(i,j)]
 * for i != j,   dV_i = sum_{j != i} g(i,j) V_j,
 *               dx   = grad_out[b][0:D] + dV_0,   dP_t = dV_{t+1}.
 * Kept in double: dV is written to dV_out ([B][N][D] double) when not null,
 * and rounded to float into grad_dense ([B][D]) / grad_pooled ([B][T][D])
 * when those are not null. */
void oracle_interact_bwd(int64_t B, int T, int D, const float *dense,
                         const float *pooled, const float *grad_out,
                         float *grad_dense, float *grad_pooled, double *dV_out)
{
    const int N = T + 1;
    const int64_t W = D + (int64_t)N * (N - 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < B; ++b) {
        const float *go = grad_out + (size_t)b * W;
        double *dv = malloc(sizeof(double) * (size_t)N * D);
        for (int i = 0; i < N; ++i) {
            for (int d = 0; d < D; ++d)
                dv[(size_t)i * D + d] = 0.0;
            for (int j = 0; j < N; ++j) {
                if (j == i)
                    continue;
                int64_t k = i < j ? tri_pos(i, j, N) : tri_pos(j, i, N);
                double g = (double)go[D + k];
                const float *vj = vec(dense, pooled, b, T, D, j);
                for (int d = 0; d < D; ++d)
                    dv[(size_t)i * D + d] += g * (double)vj[d];
            }
        }
        for (int d = 0; d < D; ++d)
            dv[d] += (double)go[d];
        if (grad_dense)
            for (int d = 0; d < D; ++d)
                grad_dense[(size_t)b * D + d] = (float)dv[d];
        if (grad_pooled)
            for (int t = 0; t < T; ++t)
                for (int d = 0; d < D; ++d)
                    grad_pooled[((size_t)b * T + t) * D + d] =
                        (float)dv[(size_t)(t + 1) * D + d];
        if (dV_out)
            memcpy(dV_out + (size_t)b * N * D, dv, sizeof(double) * (size_t)N * D);
        free(dv);
    }
}

typedef struct {
    int64_t row; /* row of table t */
    int64_t pos; /* position of the lookup in indices[] */
    int64_t b;   /* sample whose bag holds it */
    int64_t L;   /* length of that bag */
} lookup_ref;

static int cmp_lookup(const void *a, const void *b)
{
    const lookup_ref *x = a, *y = b;
    if (x->row != y->row)
        return x->row < y->row ? -1 : 1;
    if (x->pos != y->pos)
        return x->pos < y->pos ? -1 : 1;
    return x->b < y->b ? -1 : (x->b > y->b);
}

/* Steps 2-3 of the training step, per table t:  every valid lookup p of bag
 * (t,b) contributes grad(b,t) * (mean ? 1/L : 1) to its row, the lookups of a
 * row visited in original position order (sorted by (row, position)); then
 * one update of each touched row r with its gradient sum g:
 *   ADAGRAD:  A_r += sum_d g_d^2 / D;  w_r,d -= lr * g_d / (sqrt(A_r) + eps)
 *   SGD:      w_r,d -= lr * g_d
 * in double, rounded once to float.  grad(b,t) is the D doubles at
 * grad + b * grad_stride_b + (t + grad_t0) * D.  Returns the status bits. */
static int update_rows(int T, int D, float *const *tables,
                       const int64_t *num_rows, int64_t B, int64_t nnz,
                       const int64_t *indices, const int64_t *offsets, int mode,
                       const double *grad, int64_t grad_stride_b, int grad_t0,
                       int rule, float *const *accum, float lr, float eps)
{
    int status = ORACLE_OK;
    if (offsets[0] != 0 || offsets[(int64_t)T * B] != nnz)
        status |= ORACLE_BAD_OFFSETS;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int t = 0; t < T; ++t) {
        int64_t cap = 0;
        for (int64_t b = 0; b < B; ++b) {
            int64_t lo, hi;
            bag_range(offsets, (int64_t)t * B + b, nnz, &lo, &hi);
            cap += hi - lo;
        }
        lookup_ref *refs = malloc(sizeof(lookup_ref) * (size_t)(cap ? cap : 1));
        int64_t n = 0;
        for (int64_t b = 0; b < B; ++b) {
            int64_t lo, hi;
            status |= bag_range(offsets, (int64_t)t * B + b, nnz, &lo, &hi);
            for (int64_t p = lo; p < hi; ++p) {
                int64_t r = indices[p];
                if (r < 0 || r >= num_rows[t]) {
                    status |= ORACLE_INDEX_OOB;
                    continue;
                }
                refs[n].row = r;
                refs[n].pos = p;
                refs[n].b = b;
                refs[n].L = hi - lo;
                ++n;
            }
        }
        qsort(refs, (size_t)n, sizeof(lookup_ref), cmp_lookup);

        double *g = malloc(sizeof(double) * (size_t)D);
        int64_t s = 0;
        while (s < n) {
            int64_t e = s;
            for (int d = 0; d < D; ++d)
                g[d] = 0.0;
            for (; e < n && refs[e].row == refs[s].row; ++e) {
                double scale = (mode == ORACLE_MEAN) ? 1.0 / (double)refs[e].L : 1.0;
                const double *dp = grad + (size_t)refs[e].b * grad_stride_b + (size_t)(t + grad_t0) * D;
                for (int d = 0; d < D; ++d)
                    g[d] += dp[d] * scale;
            }
            int64_t r = refs[s].row;
            float *w = tables[t] + r * (int64_t)D;
            if (rule == ORACLE_SGD) {
                for (int d = 0; d < D; ++d)
                    w[d] = (float)((double)w[d] - (double)lr * g[d]);
            } else {
                double ss = 0.0;
                for (int d = 0; d < D; ++d)
                    ss += g[d] * g[d];
                double A = (double)accum[t][r] + ss / (double)D;
                double den = sqrt(A) + (double)eps;
                for (int d = 0; d < D; ++d)
                    w[d] = (float)((double)w[d] - (double)lr * g[d] / den);
                accum[t][r] = (float)A;
            }
            s = e;
        }
        free(g);
        free(refs);
    }
    return status;
}

/* One training step of the sparse path (fp32 tables only):
 *   1. dV from oracle_interact_bwd, in double; grad_dense receives dx;
 *   2-3. update_rows with dP_t = dV_{t+1} and the given rule.
 * tables[] and accum[] (Adagrad only) are updated in place.  Returns the
 * status bits.  When the offsets are malformed only the status is
 * meaningful. */
int oracle_sparse_bwd_update(int T, int D, float *const *tables,
                             const int64_t *num_rows, int64_t B, int64_t nnz,
                             const int64_t *indices, const int64_t *offsets,
                             int mode, const float *dense, const float *pooled,
                             const float *grad_out, float *grad_dense, int rule,
                             float *const *accum, float lr, float eps)
{
    const int N = T + 1;
    double *dV = malloc(sizeof(double) * (size_t)B * N * D);
    oracle_interact_bwd(B, T, D, dense, pooled, grad_out, grad_dense, NULL, dV);
    int status = update_rows(T, D, tables, num_rows, B, nnz, indices, offsets, mode,
                             dV, (int64_t)N * D, 1, rule, accum, lr, eps);
    free(dV);
    return status;
}

/* The Adagrad training step ("DLRM", robocikowo.com, "Forward pass", last
 * sentence, with the row-wise reading). */
int oracle_sparse_bwd_adagrad(int T, int D, float *const *tables,
                              const int64_t *num_rows, int64_t B, int64_t nnz,
                              const int64_t *indices, const int64_t *offsets,
                              int mode, const float *dense, const float *pooled,
                              const float *grad_out, float *grad_dense,
                              float *const *accum, float lr, float eps)
{
    return oracle_sparse_bwd_update(T, D, tables, num_rows, B, nnz, indices, offsets, mode,
                                    dense, pooled, grad_out, grad_dense, ORACLE_ADAGRAD,
                                    accum, lr, eps);
}

/* Steps 2-3 alone, from a given gradient of the pooled vectors
 * grad_pooled[B][T][D] (float, as the interaction backward writes it). */
int oracle_embbag_bwd_update(int T, int D, float *const *tables,
                             const int64_t *num_rows, int64_t B, int64_t nnz,
                             const int64_t *indices, const int64_t *offsets,
                             int mode, const float *grad_pooled, int rule,
                             float *const *accum, float lr, float eps)
{
    double *g = malloc(sizeof(double) * ((size_t)B * T * D + 1));
    for (size_t i = 0; i < (size_t)B * T * D; ++i)
        g[i] = (double)grad_pooled[i];
    int status = update_rows(T, D, tables, num_rows, B, nnz, indices, offsets, mode,
                             g, (int64_t)T * D, 0, rule, accum, lr, eps);
    free(g);
    return status;
}

/* Raw feature IDs to rows of their tables: rows[p] = raw[p] mod V_t, the ID
 * read as an unsigned 64-bit integer, t the table whose bags hold position p
 * (table-major offsets: t with offsets[t*B] <= p < offsets[(t+1)*B]).
 * Positions outside every table's range (malformed offsets) get row 0 and
 * raise ORACLE_BAD_OFFSETS.  Returns the status bits. */
int oracle_hash_indices(int T, int64_t B, int64_t nnz, const int64_t *num_rows,
                        const uint64_t *raw, const int64_t *offsets, int64_t *rows)
{
    int status = ORACLE_OK;
    if (offsets[0] != 0 || offsets[(int64_t)T * B] != nnz)
        status |= ORACLE_BAD_OFFSETS;
    for (int64_t p = 0; p < nnz; ++p)
        rows[p] = -1;
    for (int t = 0; t < T; ++t) {
        int64_t lo = offsets[(int64_t)t * B], hi = offsets[(int64_t)(t + 1) * B];
        if (lo < 0 || hi < lo || hi > nnz) {
            status |= ORACLE_BAD_OFFSETS;
            continue;
        }
        for (int64_t p = lo; p < hi; ++p)
            rows[p] = (int64_t)(raw[p] % (uint64_t)num_rows[t]);
    }
    for (int64_t p = 0; p < nnz; ++p)
        if (rows[p] < 0) {
            rows[p] = 0;
            status |= ORACLE_BAD_OFFSETS;
        }
    return status;
}
