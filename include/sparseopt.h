/*
 * sparseopt.h -- C ABI of libsparseopt: the sparse / lazy optimizer step for
 * large fp32 embedding tables on one GB300 (sm_103a).
 *
 * What is computed (page titles and sections):
 *   "Module sparse_optimizer" (optirs-gpu 0.3.2 docs)
 *     - "Sparse gradient representations": canonical COO (strictly ascending
 *       indices) and CSR (row_offsets, col_indices strictly ascending within a
 *       row, values, dense shape); lossless CSR <-> COO by lin = row*c + col.
 *     - "Sparse SGD": params[i] -= lr*grad[i] on touched coordinates only, with
 *       optional coupled weight decay and lazily applied momentum.
 *     - "Lazy Adam": LazyAdamMode::Lazy (one decay factor) and
 *       LazyAdamMode::DormancyDecay (beta^gap catch-up, gap = t - last_step[i]);
 *       bias correction by the global step t in both modes.
 *   "DiskSparseAdam (DSA)" README
 *     - "Safe Duplicate Aggregation & Sorted I/O" and step(): duplicate indices
 *       are summed and indices sorted after deduplication.
 *     - "Validated Inputs": bad indices are explicit errors.
 *
 * Conventions shared by every entry point
 *   Memory.   Every array argument is DEVICE memory owned by the caller (state,
 *             gradient, outputs, workspace, error word); the library allocates
 *             nothing and keeps no state between calls.  Arrays are dense and
 *             row-major: a table of r rows and c columns is r*c contiguous fp32.
 *             Outputs must not overlap inputs; p, m, v, buf, last_step must not
 *             overlap each other.  Any alignment is accepted; 16-byte aligned
 *             arrays with c % 4 == 0 take the 128-bit vector path.
 *   Streams.  Work is enqueued on `stream` (0 = legacy default stream) and never
 *             synchronises the host.  The library's kernels are launched with
 *             programmatic dependent launch: each may be scheduled while the
 *             kernel before it on the stream finishes, and waits for it before
 *             touching memory that kernel may use.  One read comes earlier: on a
 *             raw (non-canonical) gradient the first kernel reads the index
 *             array before that wait, and on a CSR gradient under a per-row
 *             last_step it reads the offset and column arrays (the problems it
 *             finds reach *d_err only after the wait).  That is safe when these
 *             arrays were
 *             written by a copy, a memset, an ordinary kernel launch, or any call
 *             of this library: every call that writes an output other than
 *             optimizer state and the error word (canonical indices, offsets,
 *             permutation, linear indices, converted structures, summed or
 *             gathered values) lets the next kernel start only after those
 *             writes.  It is not safe when the index array was written by a
 *             kernel of the caller's own that releases its dependents early
 *             (programmatic dependent launch), nor when an optimizer state array
 *             (p, m, v, buf, last_step) of one call is one of those arrays of
 *             the next call on the same stream.
 *   Errors.   Host-checkable problems (null pointer, negative size, bad config,
 *             t < 1, workspace too small, a size beyond a stated limit) return a
 *             non-zero sparse_status_t before anything is enqueued.  A failed
 *             launch returns SPARSE_ERR_CUDA.  Data-dependent problems (an index
 *             out of range, non-canonical "canonical" input, t <= last_step[i],
 *             a partial row under a per-row last_step) are found on the device:
 *             the code is written to *d_err (first error wins) and the step
 *             writes NO optimizer state.  *d_err is sticky: the library never
 *             clears it, and while it is non-zero every later call that is given
 *             the same d_err leaves optimizer state alone.  Zero it (e.g.
 *             cudaMemsetAsync) before first use and after handling an error.
 *             Which code is reported when one call has several problems is
 *             unspecified.  Non-state outputs (canonical arrays, conversions)
 *             are undefined when the call sets *d_err.
 *   Workspace.ws is device scratch of at least sparse_workspace_size() bytes,
 *             256-byte aligned; its contents need not be initialised and are
 *             garbage after the call; calls that run concurrently need separate
 *             workspaces.  Canonical and CSR gradients need none (ws may be NULL).
 *             A CSR Adam step with a per-row last_step (every listed row full)
 *             given ws of at least 8*(nnz/c + 1) bytes (256-byte aligned;
 *             sparse_workspace_size(nnz/c + 1, 1, r) is enough) lists the touched
 *             rows there and updates them with the row kernel, which spreads them
 *             evenly over the GPU; without it the CSR kernel walks the rows.  Any
 *             other CSR step (per-coordinate last_step, or SGD) given ws of at
 *             least 8*(nnz + 64) bytes for Adam or 4*(nnz + 64) for SGD (256-byte
 *             aligned, rows < 2^31, t < 2^31; sparse_workspace_size(nnz + 64, 1, r)
 *             is enough) records every entry's row (and last_step gap) there during
 *             the check and updates one entry per thread without re-reading
 *             last_step.
 *   Step.     t is the global step, the 1-based number of step calls so far; it
 *             is owned by the caller and is the same t for every coordinate.
 *   State.    m, v, buf start at 0 and last_step at 0 (never touched).  A
 *             coordinate is touched when it is present in the canonical sparse
 *             structure, whatever its value; nothing else is read or written.
 *   Limits.   Raw (non-canonical) input: n <= 2^30 entries, keys < 2^32.
 *             Canonical row-COO input: n < 2^31 rows, tables of at most 2^32
 *             rows (1-D: dim <= 2^32).  CSR input: no limit beyond int64.
 */
#ifndef SPARSEOPT_H
#define SPARSEOPT_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPARSE_OK = 0,
    SPARSE_ERR_INVALID_ARG = 1,        /* host: bad pointer, size, config or enum value */
    SPARSE_ERR_INDEX_OUT_OF_RANGE = 2, /* device: an index < 0 or >= its bound */
    SPARSE_ERR_NOT_CANONICAL = 3,      /* device: indices not strictly ascending, bad offsets,
                                          or a partial row under a per-row last_step */
    SPARSE_ERR_STEP_ORDER = 4,         /* device: t <= last_step of a touched coordinate */
    SPARSE_ERR_WORKSPACE = 5,          /* host: ws missing, misaligned or too small */
    SPARSE_ERR_CUDA = 6,               /* host: a CUDA launch or runtime call failed */
    SPARSE_ERR_INTERNAL = 7,           /* device: a bounded wait between thread blocks gave up */
    SPARSE_ERR_NON_FINITE = 8,         /* device: a gradient value is NaN or infinite (sparse_check_finite) */
    SPARSE_ERR_BAD_STATE = 9           /* device: a touched m is NaN/infinite or a touched v is NaN/infinite/negative
                                          (sparse_check_state) */
} sparse_status_t;

/* "Lazy Adam": LazyAdamMode::Lazy and LazyAdamMode::DormancyDecay. */
typedef enum {
    SPARSE_LAZY_ADAM_LAZY = 0,
    SPARSE_LAZY_ADAM_DORMANCY_DECAY = 1
} sparse_lazy_adam_mode_t;

/* Where last_step lives: one int64 per table row (legal only when every touch
 * covers whole rows) or one per coordinate (r*c entries). */
typedef enum {
    SPARSE_LAST_STEP_PER_ROW = 0,
    SPARSE_LAST_STEP_PER_COORD = 1
} sparse_last_step_layout_t;

typedef enum {
    SPARSE_GRAD_ROW_COO = 0, /* n listed rows, each with c values */
    SPARSE_GRAD_CSR = 1      /* CsrGradient: row_off[r+1], cols[nnz], vals[nnz] */
} sparse_grad_form_t;

/* Adam weight decay ("DiskSparseAdam (DSA)" README, "Explicit Weight Decay
 * Semantics", Euclidean case): L2 adds weight_decay*p to the gradient (classic
 * Adam L2); DECOUPLED adds weight_decay*p to the descent direction (AdamW).
 * Like every other term it acts on touched coordinates only, with the value of
 * p read at the step (no decay over dormant steps). */
typedef enum {
    SPARSE_ADAM_WD_L2 = 0,
    SPARSE_ADAM_WD_DECOUPLED = 1
} sparse_adam_wd_mode_t;

/* SparseAdamConfig.  beta1, beta2 in [0, 1); eps > 0; lr finite; weight_decay
 * >= 0 and finite (0: plain lazy Adam, whatever the mode); weight_decay_mode a
 * sparse_adam_wd_mode_t. */
typedef struct {
    double lr, beta1, beta2, eps;
    double weight_decay;
    int32_t weight_decay_mode;
} sparse_adam_config_t;

/* SparseSgdConfig.  momentum >= 0 and weight_decay >= 0, finite; lr finite. */
typedef struct {
    double lr, momentum, weight_decay;
} sparse_sgd_config_t;

/* A gradient for an (r, c) table (host struct, device arrays).
 *   ROW_COO: row_idx[n] (int64), vals[n*c] row-major.  is_canonical = 1 asserts
 *            strictly ascending rows (checked on the device); 0 = raw: any order,
 *            duplicates allowed and summed (DSA "Safe Duplicate Aggregation").
 *   CSR:     row_off[r+1] (int64, row_off[0] = 0, non-decreasing, row_off[r] = n),
 *            cols[n] (int32, strictly ascending within a row, in [0, c)), vals[n];
 *            n is nnz; always canonical (checked on the device). */
typedef struct {
    sparse_grad_form_t form;
    int64_t n;
    const int64_t* row_idx;
    const int64_t* row_off;
    const int32_t* cols;
    const float* vals;
    int is_canonical;
} sparse_grad_t;

/* Bytes of workspace a raw (non-canonical) call with n entries of width c and
 * keys < bound needs.  Covers every entry point of this header. */
size_t sparse_workspace_size(int64_t n, int64_t c, int64_t bound);

/* Static description of a status code (never NULL). */
const char* sparse_status_string(sparse_status_t status);

/*
 * sparse_canonicalize -- raw COO -> canonical COO.
 * "Sparse gradient representations" (canonical form) with the DSA duplicate
 * rule: indices sorted ascending, duplicates removed, the values of each index
 * summed.  Summation is compensated fp32 (error-free two-sum) in a fixed order,
 * so the result is deterministic and within about one rounding of the exact
 * sum; a lone value passes through bit for bit.
 *   idx[n]        int64 keys in [0, bound); bound <= 2^32
 *   vals[n*c]     fp32, row-major (c = 1 for a 1-D view)
 *   idx_out[n]    out: the U unique keys, strictly ascending (first U entries)
 *   vals_out[n*c] out: the U summed rows (may be NULL to skip the values)
 *   seg_off_out[n+1] out (may be NULL): run boundaries in the stable sorted order;
 *                 run u holds the entries seg_off_out[u] .. seg_off_out[u+1]-1
 *   perm_out[n]   out (may be NULL): the stable sorting permutation (input
 *                 position of each sorted entry)
 *   d_nnz_out     out: U, written on the device (int64)
 */
sparse_status_t sparse_canonicalize(const int64_t* idx, const float* vals, int64_t n, int64_t c,
                                    int64_t bound, int64_t* idx_out, float* vals_out,
                                    int64_t* seg_off_out, int64_t* perm_out, int64_t* d_nnz_out,
                                    void* ws, size_t ws_bytes, int32_t* d_err, cudaStream_t stream);

/*
 * sparse_csr_to_coo -- CsrGradient::to_coo ("Sparse gradient representations"):
 * lin_out[j] = row(j)*c + cols[j] for the nnz entries of an (r, c) CSR.  The
 * result is strictly ascending when the CSR is well formed (checked; *d_err).
 */
sparse_status_t sparse_csr_to_coo(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c,
                                  int64_t nnz, int64_t* lin_out, int32_t* d_err, cudaStream_t stream);

/*
 * sparse_coo_to_csr -- CsrGradient::from_coo: canonical linear COO lin[nnz]
 * (strictly ascending, < r*c; checked) -> row_off_out[r+1], cols_out[nnz] with
 * row = lin / c, col = lin % c.  The values array is shared unchanged.
 */
sparse_status_t sparse_coo_to_csr(const int64_t* lin, int64_t nnz, int64_t r, int64_t c,
                                  int64_t* row_off_out, int32_t* cols_out, int32_t* d_err,
                                  cudaStream_t stream);

/*
 * sparse_row_coo_to_csr -- canonical row-COO (rows[nrows] strictly ascending
 * in [0, r), each listing all c columns; checked) -> the same gradient as CSR:
 * row_off_out[r+1], cols_out[nrows*c].  The values array is shared unchanged.
 */
sparse_status_t sparse_row_coo_to_csr(const int64_t* rows, int64_t nrows, int64_t r, int64_t c,
                                      int64_t* row_off_out, int32_t* cols_out, int32_t* d_err,
                                      cudaStream_t stream);

/*
 * sparse_adam_step -- SparseAdam over a 1-D parameter of `dim` fp32 values
 * ("Lazy Adam").  p, m, v: [dim] fp32; last_step: [dim] int64.  idx[nnz],
 * g[nnz]: canonical (is_canonical = 1, strictly ascending) or raw (0: any
 * order, duplicates summed; needs ws).  For every touched coordinate i:
 *   gap = t - last_step[i]; b = beta (Lazy) or beta^gap (DormancyDecay);
 *   m = b1*m + (1-beta1)*g; v = b2*v + (1-beta2)*g^2;
 *   p -= lr * (m/(1-beta1^t)) / (sqrt(v/(1-beta2^t)) + eps); last_step[i] = t.
 * Arithmetic is fp32; beta^gap is exp2(gap*log2(beta)) (beta itself at gap 1).
 */
sparse_status_t sparse_adam_step(float* p, float* m, float* v, int64_t* last_step, int64_t dim,
                                 const int64_t* idx, const float* g, int64_t nnz, int is_canonical,
                                 int64_t t, sparse_adam_config_t cfg, sparse_lazy_adam_mode_t mode,
                                 void* ws, size_t ws_bytes, int32_t* d_err, cudaStream_t stream);

/*
 * sparse_adam_table_step -- SparseAdamTable over an (r, c) fp32 table, same
 * update as sparse_adam_step on every touched coordinate.  last_step holds r
 * (PER_ROW) or r*c (PER_COORD) int64 entries; PER_ROW requires whole-row
 * touches (always true for ROW_COO; checked for CSR).  The gradient is a
 * sparse_grad_t (host pointer to a host struct).
 */
sparse_status_t sparse_adam_table_step(float* p, float* m, float* v, int64_t* last_step,
                                       sparse_last_step_layout_t ls_layout, int64_t r, int64_t c,
                                       const sparse_grad_t* grad, int64_t t, sparse_adam_config_t cfg,
                                       sparse_lazy_adam_mode_t mode, void* ws, size_t ws_bytes,
                                       int32_t* d_err, cudaStream_t stream);

/*
 * sparse_sgd_step -- SparseSgd over a 1-D parameter ("Sparse SGD").  For every
 * touched coordinate: g' = g + weight_decay*p; momentum > 0: buf = momentum*buf
 * + g', p -= lr*buf; momentum = 0: p -= lr*g' (buf unused, may be NULL).
 * Momentum is lazy: untouched buffers are not decayed.
 */
sparse_status_t sparse_sgd_step(float* p, float* buf, int64_t dim, const int64_t* idx, const float* g,
                                int64_t nnz, int is_canonical, sparse_sgd_config_t cfg, void* ws,
                                size_t ws_bytes, int32_t* d_err, cudaStream_t stream);

/* sparse_sgd_table_step -- SparseSgdTable over an (r, c) fp32 table. */
sparse_status_t sparse_sgd_table_step(float* p, float* buf, int64_t r, int64_t c,
                                      const sparse_grad_t* grad, sparse_sgd_config_t cfg, void* ws,
                                      size_t ws_bytes, int32_t* d_err, cudaStream_t stream);

/*
 * sparse_check_finite -- optional validation of gradient values ("DiskSparseAdam
 * (DSA)" README, "Validated Inputs": non-finite gradients are an explicit error).
 *   vals: n fp32 values (a gradient's value array: n = entries x c for row-COO,
 *   nnz for CSR).  Any NaN or infinity sets *d_err = SPARSE_ERR_NON_FINITE.
 *   Enqueued before a step on the same stream with the same d_err, it makes that
 *   step write no state when a value is not finite (the error word is sticky).
 *   Reads the values once (4 bytes each); n = 0 is a no-op.
 */
sparse_status_t sparse_check_finite(const float* vals, int64_t n, int32_t* d_err, cudaStream_t stream);

/*
 * sparse_check_state -- optional validation of the Adam moments a step would
 * read ("DiskSparseAdam (DSA)" README, "Validated Inputs": NaN or negative
 * moment rows have explicit behaviour; here they are an explicit error).
 *   m, v:  the Adam moments of an (r, c) table (r*c fp32 each; c = 1 for a 1-D
 *          parameter of dim = r values).
 *   grad:  the gradient of the step about to run (host struct, device arrays),
 *          in either form.  ROW_COO: every column of each listed row, in any
 *          order, repeats allowed (is_canonical is ignored; a row outside [0, r)
 *          sets SPARSE_ERR_INDEX_OUT_OF_RANGE).  CSR: the listed (row, column)
 *          coordinates; the structure is validated as by the step.
 *   A touched m that is NaN or infinite, or a touched v that is NaN, infinite or
 *   below zero (-0.0 is not below zero) sets *d_err = SPARSE_ERR_BAD_STATE.
 *   Untouched coordinates are not read; nothing but *d_err is written.
 *   Enqueued before a step on the same stream with the same d_err, it makes that
 *   step write no state when a moment it would read is corrupted (the error word
 *   is sticky).  Without it, a step reads such moments as IEEE values.
 *   Reads 8 bytes per touched coordinate (per listed row for ROW_COO: repeats
 *   are read again, mostly from L2); n = 0 is a no-op.
 */
sparse_status_t sparse_check_state(const float* m, const float* v, int64_t r, int64_t c, const sparse_grad_t* grad,
                                   int32_t* d_err, cudaStream_t stream);

/*
 * sparse_read_rows -- the rows of a table at the given indices ("DiskSparseAdam
 * (DSA)" README, API read_rows(indices): the lookup that feeds the forward pass,
 * indices validated).
 *   table: r x c fp32 row-major; idx: n int64 (any order, repeats allowed);
 *   out:   n x c fp32, out[i*c + k] = table[idx[i]*c + k], copied bit for bit.
 *   An index outside [0, r) sets *d_err = SPARSE_ERR_INDEX_OUT_OF_RANGE and its
 *   output row is left unwritten (the other rows are still copied).  n = 0 is a
 *   no-op.  table and out must not overlap.
 */
sparse_status_t sparse_read_rows(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out,
                                 int32_t* d_err, cudaStream_t stream);

/*
 * sparse_canonicalize_static_ws -- sparse_canonicalize without a caller workspace
 * (no counterpart on the pages: this serves callers, not the method).
 *
 * For callers that cannot allocate device memory -- code running inside a host
 * application that owns every device allocation through its own pool, or on a
 * thread or in a runtime where cudaMalloc is not allowed -- the scratch comes
 * from one fixed device array of SPARSE_STATIC_WS_BYTES compiled into the
 * library.  Every GPU that loads the library holds that array until the process
 * exits.  The call allocates nothing (no cudaMalloc, no cudaFree).
 *   Arguments, outputs, results and errors are those of sparse_canonicalize,
 *   without ws / ws_bytes.  Inputs and outputs are still caller memory.
 *   Limit: the call needs sparse_workspace_size(n, c, bound) <= SPARSE_STATIC_WS_BYTES
 *   (for example, 65,536 entries of 256 columns fit; the exact limit depends on
 *   n, c and bound); larger calls return
 *   SPARSE_ERR_WORKSPACE before anything is enqueued.
 *   Set-up: every call looks up the array's device address on the current
 *   device (cudaGetSymbolAddress, with that device current); nothing is cached,
 *   so a device reset or a re-created primary context is picked up.  Under
 *   CUDA's lazy module loading the array itself is created by the first call on
 *   each device (when the library's device code is loaded there): that first
 *   call can fail with SPARSE_ERR_CUDA on a device with no free memory, so make
 *   it at set-up time, before any stream capture; later calls allocate nothing.
 *   Sharing: every call uses the same array, which keeps the previous call's
 *   contents (each call clears what it needs cleared).  Calls whose work
 *   overlaps on the GPU -- on different streams, or from different host threads
 *   -- race on the array and give undefined results: serialise them.
 */
#define SPARSE_STATIC_WS_BYTES (16u * 1024u * 1024u)
sparse_status_t sparse_canonicalize_static_ws(const int64_t* idx, const float* vals, int64_t n, int64_t c,
                                              int64_t bound, int64_t* idx_out, float* vals_out,
                                              int64_t* seg_off_out, int64_t* perm_out, int64_t* d_nnz_out,
                                              int32_t* d_err, cudaStream_t stream);

/*
 * Per-kernel timing (diagnostics; no counterpart on the pages).  While enabled,
 * every kernel the library enqueues is bracketed by two CUDA events on its
 * stream.  sparse_profile_read() waits for every recorded event, then reports
 * up to max_entries kernels: names[i] (static strings), launches[i] and the
 * summed GPU time total_ms[i]; it returns the number of distinct kernels seen
 * since the last reset.  Any output pointer may be NULL.  Host-side state,
 * guarded by a mutex; intended for measurement runs, not for production steps.
 */
void sparse_profile_enable(int enable);
void sparse_profile_reset(void);
int sparse_profile_read(int max_entries, const char** names, int64_t* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* SPARSEOPT_H */
