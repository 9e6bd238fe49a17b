/*
 * sparse_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, obviously correct CPU oracle for the sparse / lazy optimizer
 * step.  Only the test suite, __graft_entry__.smoke() and bench.py's CPU
 * baseline / reference arm load it.  It shares no code, header, table or helper
 * with the CUDA library; the two only ever see the same seeded inputs.
 *
 * Sources (page title, section):
 *   [S1] "Module sparse_optimizer" (optirs-gpu 0.3.2 docs), "Sparse gradient
 *        representations": canonical COO (strictly ascending indices), CSR
 *        (row_offsets, col_indices strictly ascending within a row, values,
 *        dense shape), and the lossless CSR <-> COO mapping lin = row*c + col.
 *   [S2] same page, "Sparse SGD": params[i] -= lr*grad[i] on touched i only,
 *        optional coupled weight decay and lazily applied momentum; untouched
 *        coordinates are left bit-identical.
 *   [S3] same page, "Lazy Adam", LazyAdamMode::Lazy: single decay factor.
 *   [S4] same page, LazyAdamMode::DormancyDecay: beta^gap catch-up with
 *        gap = t - last_step[i] >= 1.
 *   [S5] same page, closing paragraph of "Lazy Adam": bias correction always by
 *        the global step count t, never by a per-coordinate visit count.
 *   [S6] "DiskSparseAdam (DSA)" README, Key Features "Safe Duplicate
 *        Aggregation & Sorted I/O" and API step(): duplicate indices are summed,
 *        indices sorted after deduplication; "Validated Inputs": negative or
 *        out-of-range indices are explicit errors.
 *   [S9] same README, "Validated Inputs": non-finite gradients are an explicit
 *        error.
 *   [S8] same README, API read_rows(indices): the rows of the table at the given
 *        indices (the lookup that feeds the forward pass), indices validated.
 *   [S10] same README, "Validated Inputs": NaN or negative moment rows have an
 *        explicit, defined behaviour (here: an explicit error before any write).
 *   [S7] same README, "Explicit Weight Decay Semantics" and the API's
 *        weight_decay / weight_decay_mode (Euclidean case, k = 0):
 *        "l2" adds wd*w to the gradient (classic Adam L2); "decoupled" adds
 *        wd*w to the descent direction (AdamW).
 *
 * Readings where the pages are silent:
 *   - duplicates are summed in fp64 in input order, starting from the first
 *     value, and rounded once to fp32 (a single value passes through unchanged);
 *   - a coordinate is touched when it is present in the canonical structure,
 *     whatever its (summed) value;
 *   - m = v = buf = 0 and last_step = 0 initially, t >= 1; t <= last_step[i] is
 *     an error (code 4), not a NaN;
 *   - eps is added outside the square root of the bias-corrected v_hat, exactly
 *     as printed in [S3];
 *   - SGD momentum: buf = mu*buf + g', no dampening, no Nesterov, no mu^gap
 *     catch-up; weight decay coupled: g' = g + wd*p;
 *   - last_step is written (= t) in both Adam modes;
 *   - Adam weight decay, like every other term, acts on touched coordinates only
 *     and uses the parameter value read at the step (no decay over dormant steps).
 *
 * Arithmetic: every floating-point step in fp64.  State is read from its
 * storage type (fp32, or fp64 for the pin tests) and rounded once on store.
 * Every function validates all of its input before it writes anything, so an
 * error leaves every output and all state untouched.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
    OR_OK = 0,
    OR_ERR_INVALID_ARG = 1,
    OR_ERR_INDEX_OUT_OF_RANGE = 2,
    OR_ERR_NOT_CANONICAL = 3,
    OR_ERR_STEP_ORDER = 4,
    OR_ERR_NON_FINITE = 8,
    OR_ERR_BAD_STATE = 9,
    OR_ERR_NO_MEMORY = 100
};

enum { OR_MODE_LAZY = 0, OR_MODE_DORMANCY_DECAY = 1 };
enum { OR_WD_L2 = 0, OR_WD_DECOUPLED = 1 };
enum { OR_LS_PER_ROW = 0, OR_LS_PER_COORD = 1 };
enum { OR_FORM_ROW_COO = 0, OR_FORM_CSR = 1 };

/* ------------------------------------------------------------------ */
/* state storage: fp32 (what the optimizer keeps) or fp64 (pin tests)  */
/* ------------------------------------------------------------------ */
static double ld(const void* a, int64_t i, int is_f64)
{
    return is_f64 ? ((const double*)a)[i] : (double)((const float*)a)[i];
}

static void st(void* a, int64_t i, double x, int is_f64)
{
    if (is_f64)
        ((double*)a)[i] = x;
    else
        ((float*)a)[i] = (float)x;
}

/* ------------------------------------------------------------------ */
/* canonical form [S1], duplicate summing [S6]                          */
/* ------------------------------------------------------------------ */
typedef struct {
    int64_t key;
    int64_t pos;
} key_pos_t;

static int cmp_key_pos(const void* a, const void* b)
{
    const key_pos_t* x = (const key_pos_t*)a;
    const key_pos_t* y = (const key_pos_t*)b;
    if (x->key != y->key) return x->key < y->key ? -1 : 1;
    if (x->pos != y->pos) return x->pos < y->pos ? -1 : 1;
    return 0;
}

/*
 * Raw COO (indices in any order, duplicates allowed) -> canonical COO.
 * idx[n] in [0, bound); vals[n*c] row-major (c = 1 for a 1-D view).
 * Outputs: idx_out[U] strictly ascending, vals_out[U*c] the per-index sums,
 * seg_off_out[U+1] the run boundaries in the stably sorted order, perm_out[n]
 * (may be NULL) the stable sorting permutation, *nnz_out = U.
 * Sorting (key, position) pairs is a stable sort of the keys.
 */
int oracle_canonicalize(const int64_t* idx, const float* vals, int64_t n, int64_t c,
                        int64_t bound, int64_t* idx_out, float* vals_out,
                        int64_t* seg_off_out, int64_t* perm_out, int64_t* nnz_out)
{
    if (n < 0 || c < 1 || bound < 1) return OR_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (idx[i] < 0 || idx[i] >= bound) return OR_ERR_INDEX_OUT_OF_RANGE;

    key_pos_t* kp = (key_pos_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(key_pos_t));
    if (!kp) return OR_ERR_NO_MEMORY;
    for (int64_t i = 0; i < n; ++i) {
        kp[i].key = idx[i];
        kp[i].pos = i;
    }
    qsort(kp, (size_t)n, sizeof(key_pos_t), cmp_key_pos);

    int64_t u = 0;
    int64_t a = 0;
    while (a < n) {
        int64_t b = a + 1;
        while (b < n && kp[b].key == kp[a].key) ++b;
        idx_out[u] = kp[a].key;
        seg_off_out[u] = a;
        for (int64_t col = 0; col < c; ++col) {
            double s = (double)vals[kp[a].pos * c + col];
            for (int64_t j = a + 1; j < b; ++j) s += (double)vals[kp[j].pos * c + col];
            vals_out[u * c + col] = (float)s;
        }
        ++u;
        a = b;
    }
    seg_off_out[u] = n;
    if (perm_out)
        for (int64_t j = 0; j < n; ++j) perm_out[j] = kp[j].pos;
    *nnz_out = u;
    free(kp);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* CSR <-> COO [S1]: lin = row*c + col                                  */
/* ------------------------------------------------------------------ */

/* CSR well-formedness: row_off[0] = 0, non-decreasing, row_off[r] = nnz, every
 * column in [0, c) and strictly ascending within its row.  With full_rows set,
 * every non-empty row must list all c columns. */
int oracle_csr_validate(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c,
                        int64_t nnz, int full_rows)
{
    if (r < 0 || c < 1 || nnz < 0) return OR_ERR_INVALID_ARG;
    if (row_off[0] != 0 || row_off[r] != nnz) return OR_ERR_NOT_CANONICAL;
    for (int64_t row = 0; row < r; ++row) {
        int64_t a = row_off[row], b = row_off[row + 1];
        if (b < a) return OR_ERR_NOT_CANONICAL;
        for (int64_t j = a; j < b; ++j) {
            if (cols[j] < 0 || cols[j] >= c) return OR_ERR_INDEX_OUT_OF_RANGE;
            if (j > a && cols[j] <= cols[j - 1]) return OR_ERR_NOT_CANONICAL;
        }
        if (full_rows && b > a && b - a != c) return OR_ERR_NOT_CANONICAL;
    }
    return OR_OK;
}

int oracle_csr_to_coo(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c,
                      int64_t nnz, int64_t* lin_out)
{
    int rc = oracle_csr_validate(row_off, cols, r, c, nnz, 0);
    if (rc) return rc;
    for (int64_t row = 0; row < r; ++row)
        for (int64_t j = row_off[row]; j < row_off[row + 1]; ++j)
            lin_out[j] = row * c + (int64_t)cols[j];
    return OR_OK;
}

/* Canonical linear COO over an (r, c) table -> CSR.  Offsets are the running
 * count of entries per row (count, then prefix sum). */
int oracle_coo_to_csr(const int64_t* lin, int64_t nnz, int64_t r, int64_t c,
                      int64_t* row_off_out, int32_t* cols_out)
{
    if (nnz < 0 || r < 0 || c < 1) return OR_ERR_INVALID_ARG;
    for (int64_t j = 0; j < nnz; ++j) {
        if (lin[j] < 0 || lin[j] >= r * c) return OR_ERR_INDEX_OUT_OF_RANGE;
        if (j > 0 && lin[j] <= lin[j - 1]) return OR_ERR_NOT_CANONICAL;
    }
    for (int64_t i = 0; i <= r; ++i) row_off_out[i] = 0;
    for (int64_t j = 0; j < nnz; ++j) {
        int64_t row = lin[j] / c;
        cols_out[j] = (int32_t)(lin[j] - row * c);
        row_off_out[row + 1] += 1;
    }
    for (int64_t i = 0; i < r; ++i) row_off_out[i + 1] += row_off_out[i];
    return OR_OK;
}

/* Canonical row-COO (strictly ascending rows, each a full row of c values) ->
 * CSR over the same (r, c) table.  The values array is unchanged. */
int oracle_row_coo_to_csr(const int64_t* rows, int64_t nrows, int64_t r, int64_t c,
                          int64_t* row_off_out, int32_t* cols_out)
{
    if (nrows < 0 || r < 0 || c < 1) return OR_ERR_INVALID_ARG;
    for (int64_t u = 0; u < nrows; ++u) {
        if (rows[u] < 0 || rows[u] >= r) return OR_ERR_INDEX_OUT_OF_RANGE;
        if (u > 0 && rows[u] <= rows[u - 1]) return OR_ERR_NOT_CANONICAL;
    }
    for (int64_t i = 0; i <= r; ++i) row_off_out[i] = 0;
    for (int64_t u = 0; u < nrows; ++u) {
        row_off_out[rows[u] + 1] = c;
        for (int64_t k = 0; k < c; ++k) cols_out[u * c + k] = (int32_t)k;
    }
    for (int64_t i = 0; i < r; ++i) row_off_out[i + 1] += row_off_out[i];
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* the touched-coordinate list of one step                             */
/* ------------------------------------------------------------------ */
typedef struct {
    int64_t k;      /* number of touched coordinates */
    int64_t* lin;   /* [k] linear coordinate row*c + col, strictly ascending */
    int64_t* row;   /* [k] row of each coordinate */
    float* g;       /* [k] gradient value of each coordinate (canonical, fp32) */
} touched_t;

static void touched_free(touched_t* t)
{
    free(t->lin);
    free(t->row);
    free(t->g);
}

/*
 * Builds the canonical list of touched coordinates of a step from either
 * gradient form.  Row-COO: row_idx[n] with vals[n*c]; raw input (is_canonical
 * = 0) is canonicalised first [S6]; canonical input must list strictly
 * ascending rows [S1].  CSR: row_off[r+1], cols[nnz], vals[nnz] [S1].
 */
static int build_touched(int64_t r, int64_t c, int form, const int64_t* row_idx, int64_t n,
                         int is_canonical, const int64_t* row_off, const int32_t* cols,
                         const float* vals, int full_rows, touched_t* out)
{
    memset(out, 0, sizeof(*out));
    if (form == OR_FORM_ROW_COO) {
        if (n < 0) return OR_ERR_INVALID_ARG;
        const int64_t* rows = row_idx;
        const float* gv = vals;
        int64_t nr = n;
        int64_t* crow = NULL;
        float* cval = NULL;
        int64_t* seg = NULL;
        if (!is_canonical) {
            crow = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
            cval = (float*)malloc((size_t)(n > 0 ? n : 1) * (size_t)c * sizeof(float));
            seg = (int64_t*)malloc((size_t)(n + 1) * sizeof(int64_t));
            if (!crow || !cval || !seg) {
                free(crow); free(cval); free(seg);
                return OR_ERR_NO_MEMORY;
            }
            int rc = oracle_canonicalize(row_idx, vals, n, c, r > 0 ? r : 1, crow, cval, seg, NULL, &nr);
            if (rc == OR_OK && r == 0 && n > 0) rc = OR_ERR_INDEX_OUT_OF_RANGE;
            if (rc) {
                free(crow); free(cval); free(seg);
                return rc;
            }
            rows = crow;
            gv = cval;
        } else {
            for (int64_t u = 0; u < n; ++u) {
                if (rows[u] < 0 || rows[u] >= r) return OR_ERR_INDEX_OUT_OF_RANGE;
                if (u > 0 && rows[u] <= rows[u - 1]) return OR_ERR_NOT_CANONICAL;
            }
        }
        int64_t k = nr * c;
        out->k = k;
        out->lin = (int64_t*)malloc((size_t)(k > 0 ? k : 1) * sizeof(int64_t));
        out->row = (int64_t*)malloc((size_t)(k > 0 ? k : 1) * sizeof(int64_t));
        out->g = (float*)malloc((size_t)(k > 0 ? k : 1) * sizeof(float));
        if (!out->lin || !out->row || !out->g) {
            touched_free(out);
            free(crow); free(cval); free(seg);
            return OR_ERR_NO_MEMORY;
        }
        for (int64_t u = 0; u < nr; ++u)
            for (int64_t col = 0; col < c; ++col) {
                out->lin[u * c + col] = rows[u] * c + col;
                out->row[u * c + col] = rows[u];
                out->g[u * c + col] = gv[u * c + col];
            }
        free(crow); free(cval); free(seg);
        return OR_OK;
    }
    if (form == OR_FORM_CSR) {
        int rc = oracle_csr_validate(row_off, cols, r, c, n, full_rows);
        if (rc) return rc;
        out->k = n;
        out->lin = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
        out->row = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
        out->g = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
        if (!out->lin || !out->row || !out->g) {
            touched_free(out);
            return OR_ERR_NO_MEMORY;
        }
        rc = oracle_csr_to_coo(row_off, cols, r, c, n, out->lin);
        for (int64_t row = 0; row < r; ++row)
            for (int64_t j = row_off[row]; j < row_off[row + 1]; ++j) {
                out->row[j] = row;
                out->g[j] = vals[j];
            }
        return rc;
    }
    return OR_ERR_INVALID_ARG;
}

/* ------------------------------------------------------------------ */
/* lazy Adam [S3] [S4] [S5]                                             */
/* ------------------------------------------------------------------ */

/*
 * One lazy Adam step over an (r, c) table.  p, m, v hold r*c values of type
 * fp32 (state_f64 = 0) or fp64 (state_f64 = 1); last_step holds r (per-row) or
 * r*c (per-coordinate) int64 entries.  A per-row last_step requires that every
 * touched row is touched in all c columns.  For each touched coordinate i with
 * gradient g, at global step t:
 *     gap = t - last_step[i]                             (>= 1, [S4])
 *     b1, b2 = beta1, beta2                              (Lazy, [S3])
 *     b1, b2 = beta1^gap, beta2^gap                      (DormancyDecay, [S4])
 *     g  = g + wd*p                                      (wd_mode l2, [S7])
 *     m = b1*m + (1-beta1)*g ;  v = b2*v + (1-beta2)*g^2
 *     m_hat = m / (1 - beta1^t) ;  v_hat = v / (1 - beta2^t)     ([S5])
 *     p -= lr * m_hat / (sqrt(v_hat) + eps)                       (l2)
 *     p -= lr * (m_hat / (sqrt(v_hat) + eps) + wd*p)              (wd_mode decoupled, [S7])
 *     last_step[i] = t
 * with p on the right the value read at the step; wd = 0 is plain lazy Adam.
 * Untouched coordinates are not read or written.
 */
int oracle_adam_table_step(void* p, void* m, void* v, int state_f64, int64_t* last_step,
                           int ls_layout, int64_t r, int64_t c, int form,
                           const int64_t* row_idx, int64_t n, int is_canonical,
                           const int64_t* row_off, const int32_t* cols, const float* vals,
                           int64_t t, double lr, double beta1, double beta2, double eps, int mode,
                           double weight_decay, int wd_mode)
{
    if (r < 0 || c < 1 || t < 1) return OR_ERR_INVALID_ARG;
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0)) return OR_ERR_INVALID_ARG;
    if (!(eps > 0.0) || !isfinite(eps) || !isfinite(lr)) return OR_ERR_INVALID_ARG;
    if (mode != OR_MODE_LAZY && mode != OR_MODE_DORMANCY_DECAY) return OR_ERR_INVALID_ARG;
    if (ls_layout != OR_LS_PER_ROW && ls_layout != OR_LS_PER_COORD) return OR_ERR_INVALID_ARG;
    if (!(weight_decay >= 0.0) || !isfinite(weight_decay)) return OR_ERR_INVALID_ARG;
    if (wd_mode != OR_WD_L2 && wd_mode != OR_WD_DECOUPLED) return OR_ERR_INVALID_ARG;

    touched_t tc;
    int rc = build_touched(r, c, form, row_idx, n, is_canonical, row_off, cols, vals,
                           ls_layout == OR_LS_PER_ROW, &tc);
    if (rc) {
        touched_free(&tc);
        return rc;
    }
    /* every touched coordinate must have last_step < t before anything is written */
    for (int64_t k = 0; k < tc.k; ++k) {
        int64_t s = last_step[ls_layout == OR_LS_PER_ROW ? tc.row[k] : tc.lin[k]];
        if (s >= t) {
            touched_free(&tc);
            return OR_ERR_STEP_ORDER;
        }
    }
    const double bc1 = 1.0 - pow(beta1, (double)t);
    const double bc2 = 1.0 - pow(beta2, (double)t);
    for (int64_t k = 0; k < tc.k; ++k) {
        const int64_t i = tc.lin[k];
        const int64_t s = last_step[ls_layout == OR_LS_PER_ROW ? tc.row[k] : i];
        const int64_t gap = t - s;
        const double p0 = ld(p, i, state_f64);
        double g = (double)tc.g[k];
        if (wd_mode == OR_WD_L2) g += weight_decay * p0;
        double b1 = beta1, b2 = beta2;
        if (mode == OR_MODE_DORMANCY_DECAY) {
            b1 = pow(beta1, (double)gap);
            b2 = pow(beta2, (double)gap);
        }
        const double mi = b1 * ld(m, i, state_f64) + (1.0 - beta1) * g;
        const double vi = b2 * ld(v, i, state_f64) + (1.0 - beta2) * g * g;
        const double m_hat = mi / bc1;
        const double v_hat = vi / bc2;
        double dir = m_hat / (sqrt(v_hat) + eps);
        if (wd_mode == OR_WD_DECOUPLED) dir += weight_decay * p0;
        const double pi = p0 - lr * dir;
        st(m, i, mi, state_f64);
        st(v, i, vi, state_f64);
        st(p, i, pi, state_f64);
        if (ls_layout == OR_LS_PER_COORD) last_step[i] = t;
    }
    /* per-row last_step: written after every coordinate of the step has read it */
    if (ls_layout == OR_LS_PER_ROW)
        for (int64_t k = 0; k < tc.k; ++k) last_step[tc.row[k]] = t;
    touched_free(&tc);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* lazy SGD [S2]                                                        */
/* ------------------------------------------------------------------ */

/*
 * One sparse SGD step over an (r, c) table.  For each touched coordinate i:
 *     g'  = g + wd * p[i]                (coupled weight decay)
 *     buf = mu * buf[i] + g'   ;  p[i] -= lr * buf     (momentum > 0)
 *     p[i] -= lr * g'                                   (momentum = 0; buf unused, may be NULL)
 * Untouched coordinates (and their momentum buffers) are not read or written.
 */
int oracle_sgd_table_step(void* p, void* buf, int state_f64, int64_t r, int64_t c, int form,
                          const int64_t* row_idx, int64_t n, int is_canonical,
                          const int64_t* row_off, const int32_t* cols, const float* vals,
                          double lr, double momentum, double weight_decay)
{
    if (r < 0 || c < 1) return OR_ERR_INVALID_ARG;
    if (!isfinite(lr) || !(momentum >= 0.0) || !isfinite(momentum)) return OR_ERR_INVALID_ARG;
    if (!(weight_decay >= 0.0) || !isfinite(weight_decay)) return OR_ERR_INVALID_ARG;
    if (momentum != 0.0 && buf == NULL) return OR_ERR_INVALID_ARG;
    touched_t tc;
    int rc = build_touched(r, c, form, row_idx, n, is_canonical, row_off, cols, vals, 0, &tc);
    if (rc) {
        touched_free(&tc);
        return rc;
    }
    for (int64_t k = 0; k < tc.k; ++k) {
        const int64_t i = tc.lin[k];
        const double pi = ld(p, i, state_f64);
        const double gd = (double)tc.g[k] + weight_decay * pi;
        if (momentum != 0.0) {
            const double bi = momentum * ld(buf, i, state_f64) + gd;
            st(buf, i, bi, state_f64);
            st(p, i, pi - lr * bi, state_f64);
        } else {
            st(p, i, pi - lr * gd, state_f64);
        }
    }
    touched_free(&tc);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* row gather [S8]                                                     */
/* ------------------------------------------------------------------ */

/*
 * out[i*c .. i*c + c) = table[idx[i]*c .. idx[i]*c + c) for i < n, copied value by
 * value (bit for bit).  Every index is checked first (0 <= idx[i] < r); on a bad
 * index nothing is written.
 */
int oracle_read_rows(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out)
{
    if (r < 0 || c < 1 || n < 0) return OR_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (idx[i] < 0 || idx[i] >= r) return OR_ERR_INDEX_OUT_OF_RANGE;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t k = 0; k < c; ++k) out[i * c + k] = table[idx[i] * c + k];
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* gradient validation [S9]                                            */
/* ------------------------------------------------------------------ */

/* OR_ERR_NON_FINITE when any of the n values is NaN or infinite, else OK. */
int oracle_check_finite(const float* vals, int64_t n)
{
    if (n < 0) return OR_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (!isfinite(vals[i])) return OR_ERR_NON_FINITE;
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* moment-state validation [S10]                                        */
/* ------------------------------------------------------------------ */

/*
 * Checks the Adam moments a step with this gradient would read.  The touched
 * coordinates are every column of each listed row (row-COO: row_idx[n], any
 * order, repeats allowed) or the listed (row, cols[j]) pairs (CSR: row_off[r+1],
 * cols[n], validated like a CSR gradient).  Returns
 *   OR_ERR_INDEX_OUT_OF_RANGE  a listed row outside [0, r),
 *   OR_ERR_BAD_STATE           a touched m that is NaN or infinite, or a touched
 *                              v that is NaN, infinite or below zero (-0.0 is
 *                              not below zero),
 *   OR_OK                      otherwise.
 * Untouched coordinates are never read.  Nothing is written.
 */
int oracle_check_state(const float* m, const float* v, int64_t r, int64_t c, int form,
                       const int64_t* row_idx, int64_t n, const int64_t* row_off, const int32_t* cols)
{
    if (r < 0 || c < 1 || n < 0) return OR_ERR_INVALID_ARG;
    if (form == OR_FORM_ROW_COO) {
        for (int64_t i = 0; i < n; ++i)
            if (row_idx[i] < 0 || row_idx[i] >= r) return OR_ERR_INDEX_OUT_OF_RANGE;
        for (int64_t i = 0; i < n; ++i)
            for (int64_t col = 0; col < c; ++col) {
                const int64_t k = row_idx[i] * c + col;
                if (!isfinite(m[k]) || !isfinite(v[k]) || v[k] < 0.0f) return OR_ERR_BAD_STATE;
            }
        return OR_OK;
    }
    if (form == OR_FORM_CSR) {
        const int rc = oracle_csr_validate(row_off, cols, r, c, n, 0);
        if (rc) return rc;
        for (int64_t row = 0; row < r; ++row)
            for (int64_t j = row_off[row]; j < row_off[row + 1]; ++j) {
                const int64_t k = row * c + cols[j];
                if (!isfinite(m[k]) || !isfinite(v[k]) || v[k] < 0.0f) return OR_ERR_BAD_STATE;
            }
        return OR_OK;
    }
    return OR_ERR_INVALID_ARG;
}
