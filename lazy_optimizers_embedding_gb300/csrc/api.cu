// api.cu -- the extern "C" entry points of libsparseopt (declared in
// include/sparseopt.h).  Host side only: argument validation, the per-call
// scalars (computed once in fp64, passed to the kernels in fp32), workspace
// carving and the launch sequence of each path.  No host synchronisation.
#include <cmath>
#include <cstdint>

#include "common.cuh"

namespace {

using namespace so;

constexpr int64_t kMaxRawN = int64_t(1) << 30;
constexpr int64_t kMaxCanonN = (int64_t(1) << 31) - 1;   // canonical row-COO rows (32-bit positions)
constexpr int64_t kMaxRawBound = int64_t(1) << 32;   // raw keys, and rows of a canonical row-COO table

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite(double x) { return std::isfinite(x); }

sparse_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? SPARSE_OK : SPARSE_ERR_CUDA; }

bool valid_adam_cfg(const sparse_adam_config_t& c)
{
    return finite(c.lr) && c.beta1 >= 0.0 && c.beta1 < 1.0 && c.beta2 >= 0.0 && c.beta2 < 1.0 &&
           c.eps > 0.0 && finite(c.eps) && finite(c.weight_decay) && c.weight_decay >= 0.0 &&
           (c.weight_decay_mode == SPARSE_ADAM_WD_L2 || c.weight_decay_mode == SPARSE_ADAM_WD_DECOUPLED);
}

bool valid_sgd_cfg(const sparse_sgd_config_t& c)
{
    return finite(c.lr) && finite(c.momentum) && c.momentum >= 0.0 && finite(c.weight_decay) &&
           c.weight_decay >= 0.0;
}

// Per-call scalars of "Lazy Adam": bias corrections by the global step t,
// 1 - beta, log2(beta) for the beta^gap catch-up.
AdamParams adam_params(float* p, float* m, float* v, int64_t* ls, int ls_per_coord, int64_t t,
                       const sparse_adam_config_t& cfg, sparse_lazy_adam_mode_t mode)
{
    AdamParams P{};
    P.p = p;
    P.m = m;
    P.v = v;
    P.ls = ls;
    P.ls_per_coord = ls_per_coord;
    P.dd = (mode == SPARSE_LAZY_ADAM_DORMANCY_DECAY);
    P.t = t;
    P.beta1 = static_cast<float>(cfg.beta1);
    P.beta2 = static_cast<float>(cfg.beta2);
    P.wd = static_cast<float>(cfg.weight_decay);
    P.wd_lo = static_cast<float>(cfg.weight_decay - static_cast<double>(P.wd));
    P.wd_decoupled = (cfg.weight_decay_mode == SPARSE_ADAM_WD_DECOUPLED);
    P.omb1 = static_cast<float>(1.0 - cfg.beta1);
    P.omb2 = static_cast<float>(1.0 - cfg.beta2);
    P.log2b1 = cfg.beta1 > 0.0 ? static_cast<float>(std::log2(cfg.beta1)) : -INFINITY;
    P.log2b2 = cfg.beta2 > 0.0 ? static_cast<float>(std::log2(cfg.beta2)) : -INFINITY;
    P.inv_bc1 = static_cast<float>(1.0 / (1.0 - std::pow(cfg.beta1, static_cast<double>(t))));
    P.inv_bc2 = static_cast<float>(1.0 / (1.0 - std::pow(cfg.beta2, static_cast<double>(t))));
    P.lr = static_cast<float>(cfg.lr);
    P.eps = static_cast<float>(cfg.eps);
    return P;
}

SgdParams sgd_params(float* p, float* buf, const sparse_sgd_config_t& cfg)
{
    SgdParams P{};
    P.p = p;
    P.buf = cfg.momentum != 0.0 ? buf : nullptr;  // without momentum the buffer is neither read nor written
    P.lr = static_cast<float>(cfg.lr);
    P.momentum = static_cast<float>(cfg.momentum);
    P.momentum_lo = static_cast<float>(cfg.momentum - static_cast<double>(P.momentum));
    P.wd = static_cast<float>(cfg.weight_decay);
    P.wd_lo = static_cast<float>(cfg.weight_decay - static_cast<double>(P.wd));
    return P;
}

sparse_status_t check_ws(int64_t n, int64_t c, int64_t bound, void* ws, size_t ws_bytes, WsLayout& L)
{
    L = ws_layout(n, c, bound);
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < L.total)
        return SPARSE_ERR_WORKSPACE;
    return SPARSE_OK;
}

// Per-entry scratch of the flat CSR update: `arrays` int32 arrays of nnz entries,
// each starting 256-byte aligned; rows must fit int32.
int64_t flat_stride(int64_t nnz) { return (nnz + 63) / 64 * 64; }
bool flat_fits(const void* ws, size_t ws_bytes, int64_t nnz, int64_t r, int arrays)
{
    return ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 && r <= INT32_MAX &&
           ws_bytes >= sizeof(int32_t) * static_cast<size_t>(flat_stride(nnz)) * static_cast<size_t>(arrays);
}

// Common validation of a gradient descriptor against an (r, c) table.
sparse_status_t check_grad(const sparse_grad_t* g, int64_t r, int64_t c)
{
    if (g == nullptr || r < 0 || c < 1 || g->n < 0) return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && c > INT64_MAX / r) return SPARSE_ERR_INVALID_ARG;
    if (g->form == SPARSE_GRAD_ROW_COO) {
        if (g->n > 0 && (g->row_idx == nullptr || g->vals == nullptr)) return SPARSE_ERR_INVALID_ARG;
        if (!g->is_canonical && (g->n > kMaxRawN || r > kMaxRawBound)) return SPARSE_ERR_INVALID_ARG;
        if (g->is_canonical && (g->n > kMaxCanonN || r > kMaxRawBound)) return SPARSE_ERR_INVALID_ARG;
        return SPARSE_OK;
    }
    if (g->form == SPARSE_GRAD_CSR) {
        if (g->row_off == nullptr) return SPARSE_ERR_INVALID_ARG;
        if (g->n > 0 && (g->cols == nullptr || g->vals == nullptr)) return SPARSE_ERR_INVALID_ARG;
        if (c > INT32_MAX) return SPARSE_ERR_INVALID_ARG;
        return SPARSE_OK;
    }
    return SPARSE_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

size_t sparse_workspace_size(int64_t n, int64_t c, int64_t bound)
{
    if (n < 0 || c < 1 || bound < 1) return 0;
    return ws_layout(n, c, bound).total;
}

const char* sparse_status_string(sparse_status_t status)
{
    switch (status) {
    case SPARSE_OK: return "ok";
    case SPARSE_ERR_INVALID_ARG: return "invalid argument";
    case SPARSE_ERR_INDEX_OUT_OF_RANGE: return "index out of range";
    case SPARSE_ERR_NOT_CANONICAL: return "gradient not in canonical form";
    case SPARSE_ERR_STEP_ORDER: return "global step t not greater than last_step of a touched coordinate";
    case SPARSE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPARSE_ERR_CUDA: return "CUDA error";
    case SPARSE_ERR_INTERNAL: return "internal: a bounded device wait gave up";
    case SPARSE_ERR_NON_FINITE: return "a gradient value is NaN or infinite";
    case SPARSE_ERR_BAD_STATE: return "a touched moment is NaN or infinite, or a touched second moment is negative";
    }
    return "unknown status";
}

sparse_status_t sparse_canonicalize(const int64_t* idx, const float* vals, int64_t n, int64_t c, int64_t bound,
                                    int64_t* idx_out, float* vals_out, int64_t* seg_off_out, int64_t* perm_out,
                                    int64_t* d_nnz_out, void* ws, size_t ws_bytes, int32_t* d_err,
                                    cudaStream_t stream)
{
    if (n < 0 || c < 1 || bound < 1 || bound > kMaxRawBound || n > kMaxRawN || d_err == nullptr ||
        d_nnz_out == nullptr)
        return SPARSE_ERR_INVALID_ARG;
    if (n > 0 && (idx == nullptr || idx_out == nullptr || (vals_out != nullptr && vals == nullptr)))
        return SPARSE_ERR_INVALID_ARG;
    if (n == 0) {
        if (seg_off_out) {
            cudaError_t e = cudaMemsetAsync(seg_off_out, 0, sizeof(int64_t), stream);
            if (e != cudaSuccess) return SPARSE_ERR_CUDA;
        }
        return from_cuda(cudaMemsetAsync(d_nnz_out, 0, sizeof(int64_t), stream));
    }
    WsLayout L;
    sparse_status_t st = check_ws(n, c, bound, ws, ws_bytes, L);
    if (st) return st;
    SortWs w = carve(L, ws);
    cudaError_t e = sort_and_segment(idx, n, c, bound, L, w, idx_out, seg_off_out, perm_out, d_nnz_out,
                                     nullptr, 0, 0, d_err, stream);
    if (e != cudaSuccess) return SPARSE_ERR_CUDA;
    if (vals_out) {
        const int vec4 = (c % 4 == 0) && aligned16(vals) && aligned16(vals_out);
        e = fused_rows_store_sorted(w, L, vals, c, StoreParams{vals_out}, vec4, d_err, stream);
    }
    return from_cuda(e);
}

sparse_status_t sparse_csr_to_coo(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                                  int64_t* lin_out, int32_t* d_err, cudaStream_t stream)
{
    if (r < 0 || c < 1 || c > INT32_MAX || nnz < 0 || row_off == nullptr || d_err == nullptr)
        return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && c > INT64_MAX / r) return SPARSE_ERR_INVALID_ARG;
    if (nnz > 0 && (cols == nullptr || lin_out == nullptr)) return SPARSE_ERR_INVALID_ARG;
    cudaError_t e = csr_check(row_off, cols, r, c, nnz, 0, nullptr, 0, 0, nullptr, nullptr, nullptr, d_err, stream);
    if (e == cudaSuccess && nnz > 0) e = csr_to_coo(row_off, cols, r, c, nnz, lin_out, d_err, stream);
    return from_cuda(e);
}

sparse_status_t sparse_coo_to_csr(const int64_t* lin, int64_t nnz, int64_t r, int64_t c, int64_t* row_off_out,
                                  int32_t* cols_out, int32_t* d_err, cudaStream_t stream)
{
    if (r < 0 || c < 1 || c > INT32_MAX || nnz < 0 || row_off_out == nullptr || d_err == nullptr)
        return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && c > INT64_MAX / r) return SPARSE_ERR_INVALID_ARG;
    if (nnz > 0 && (lin == nullptr || cols_out == nullptr)) return SPARSE_ERR_INVALID_ARG;
    return from_cuda(coo_to_csr(lin, nnz, r, c, row_off_out, cols_out, d_err, stream));
}

sparse_status_t sparse_row_coo_to_csr(const int64_t* rows, int64_t nrows, int64_t r, int64_t c,
                                      int64_t* row_off_out, int32_t* cols_out, int32_t* d_err,
                                      cudaStream_t stream)
{
    if (r < 0 || c < 1 || c > INT32_MAX || nrows < 0 || row_off_out == nullptr || d_err == nullptr)
        return SPARSE_ERR_INVALID_ARG;
    if (nrows > 0 && (rows == nullptr || cols_out == nullptr || c > INT64_MAX / nrows))
        return SPARSE_ERR_INVALID_ARG;
    return from_cuda(row_coo_to_csr(rows, nrows, r, c, row_off_out, cols_out, d_err, stream));
}

sparse_status_t sparse_adam_table_step(float* p, float* m, float* v, int64_t* last_step,
                                       sparse_last_step_layout_t ls_layout, int64_t r, int64_t c,
                                       const sparse_grad_t* grad, int64_t t, sparse_adam_config_t cfg,
                                       sparse_lazy_adam_mode_t mode, void* ws, size_t ws_bytes, int32_t* d_err,
                                       cudaStream_t stream)
{
    sparse_status_t st = check_grad(grad, r, c);
    if (st) return st;
    if (t < 1 || !valid_adam_cfg(cfg) || d_err == nullptr) return SPARSE_ERR_INVALID_ARG;
    if (mode != SPARSE_LAZY_ADAM_LAZY && mode != SPARSE_LAZY_ADAM_DORMANCY_DECAY) return SPARSE_ERR_INVALID_ARG;
    if (ls_layout != SPARSE_LAST_STEP_PER_ROW && ls_layout != SPARSE_LAST_STEP_PER_COORD)
        return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && (p == nullptr || m == nullptr || v == nullptr || last_step == nullptr))
        return SPARSE_ERR_INVALID_ARG;
    const int per_coord = (ls_layout == SPARSE_LAST_STEP_PER_COORD);
    const AdamParams P = adam_params(p, m, v, last_step, per_coord, t, cfg, mode);
    const int64_t n = grad->n;
    cudaError_t e = cudaSuccess;

    if (grad->form == SPARSE_GRAD_CSR) {
        // Per-row last_step: every listed row is full, so with scratch for the list of
        // listed rows (filled by the check) the gradient is a canonical row-COO over the
        // CSR's own values and takes the row kernel; otherwise the CSR kernel.
        const int64_t nrows = n / c;
        const bool as_rows = !per_coord && n > 0 && ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u) == 0 &&
                             ws_bytes >= sizeof(int64_t) * static_cast<size_t>(nrows + 1) && nrows <= kMaxCanonN &&
                             r <= kMaxRawBound;
        int64_t* rows_list = as_rows ? static_cast<int64_t*>(ws) : nullptr;
        // Per-coordinate last_step: with scratch for every entry's row and gap (filled by
        // the check), the update is one entry per thread and does not read last_step.
        int32_t *ent_row = nullptr, *ent_gap = nullptr;
        if (per_coord && n > 0 && t <= INT32_MAX && flat_fits(ws, ws_bytes, n, r, 2)) {
            ent_row = static_cast<int32_t*>(ws);
            ent_gap = ent_row + flat_stride(n);
        }
        e = csr_check(grad->row_off, grad->cols, r, c, n, !per_coord, last_step, per_coord, t, rows_list, ent_row,
                      ent_gap, d_err, stream);
        if (e == cudaSuccess && as_rows) {
            const int vec4 = (c % 4 == 0) && aligned16(p) && aligned16(m) && aligned16(v) && aligned16(grad->vals);
            e = fused_rows_adam_canon(rows_list, nrows, grad->vals, c, P, vec4, d_err, stream);
        } else if (e == cudaSuccess && ent_row) {
            e = csr_adam_flat(grad->cols, grad->vals, ent_row, ent_gap, c, n, P, d_err, stream);
        } else if (e == cudaSuccess && n > 0) {
            e = csr_adam(grad->row_off, grad->cols, grad->vals, r, c, n, P, d_err, stream);
        }
        return from_cuda(e);
    }
    if (n == 0) return SPARSE_OK;
    const int vec4 = (c % 4 == 0) && aligned16(p) && aligned16(m) && aligned16(v) && aligned16(grad->vals);
    if (grad->is_canonical) {
        e = check_canonical_rows(grad->row_idx, n, r, c, last_step, per_coord, t, d_err, stream);
        if (e == cudaSuccess) e = fused_rows_adam_canon(grad->row_idx, n, grad->vals, c, P, vec4, d_err, stream);
        return from_cuda(e);
    }
    WsLayout L;
    st = check_ws(n, c, r, ws, ws_bytes, L);
    if (st) return st;
    SortWs w = carve(L, ws);
    e = sort_and_segment(grad->row_idx, n, c, r, L, w, nullptr, nullptr, nullptr, nullptr, last_step, per_coord, t,
                         d_err, stream);
    if (e == cudaSuccess) e = fused_rows_adam_sorted(w, L, grad->vals, c, P, vec4, d_err, stream);
    return from_cuda(e);
}

sparse_status_t sparse_adam_step(float* p, float* m, float* v, int64_t* last_step, int64_t dim, const int64_t* idx,
                                 const float* g, int64_t nnz, int is_canonical, int64_t t, sparse_adam_config_t cfg,
                                 sparse_lazy_adam_mode_t mode, void* ws, size_t ws_bytes, int32_t* d_err,
                                 cudaStream_t stream)
{
    sparse_grad_t grad{};
    grad.form = SPARSE_GRAD_ROW_COO;
    grad.n = nnz;
    grad.row_idx = idx;
    grad.vals = g;
    grad.is_canonical = is_canonical;
    return sparse_adam_table_step(p, m, v, last_step, SPARSE_LAST_STEP_PER_ROW, dim, 1, &grad, t, cfg, mode, ws,
                                  ws_bytes, d_err, stream);
}

sparse_status_t sparse_sgd_table_step(float* p, float* buf, int64_t r, int64_t c, const sparse_grad_t* grad,
                                      sparse_sgd_config_t cfg, void* ws, size_t ws_bytes, int32_t* d_err,
                                      cudaStream_t stream)
{
    sparse_status_t st = check_grad(grad, r, c);
    if (st) return st;
    if (!valid_sgd_cfg(cfg) || d_err == nullptr) return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && (p == nullptr || (cfg.momentum != 0.0 && buf == nullptr))) return SPARSE_ERR_INVALID_ARG;
    const SgdParams P = sgd_params(p, buf, cfg);
    const int64_t n = grad->n;
    cudaError_t e = cudaSuccess;
    if (grad->form == SPARSE_GRAD_CSR) {
        // with scratch for every entry's row (filled by the check), one entry per thread
        int32_t* ent_row = (n > 0 && flat_fits(ws, ws_bytes, n, r, 1)) ? static_cast<int32_t*>(ws) : nullptr;
        e = csr_check(grad->row_off, grad->cols, r, c, n, 0, nullptr, 0, 0, nullptr, ent_row, nullptr, d_err, stream);
        if (e == cudaSuccess && ent_row)
            e = csr_sgd_flat(grad->cols, grad->vals, ent_row, c, n, P, d_err, stream);
        else if (e == cudaSuccess && n > 0)
            e = csr_sgd(grad->row_off, grad->cols, grad->vals, r, c, n, P, d_err, stream);
        return from_cuda(e);
    }
    if (n == 0) return SPARSE_OK;
    const int vec4 = (c % 4 == 0) && aligned16(p) && (buf == nullptr || aligned16(buf)) && aligned16(grad->vals);
    if (grad->is_canonical) {
        if (c == 1 && n <= kSmallCanonMax)   // check and update in one launch
            return from_cuda(small_canon_sgd(grad->row_idx, n, r, grad->vals, P, d_err, stream));
        e = check_canonical_rows(grad->row_idx, n, r, c, nullptr, 0, 0, d_err, stream);
        if (e == cudaSuccess) e = fused_rows_sgd_canon(grad->row_idx, n, grad->vals, c, P, vec4, d_err, stream);
        return from_cuda(e);
    }
    WsLayout L;
    st = check_ws(n, c, r, ws, ws_bytes, L);
    if (st) return st;
    SortWs w = carve(L, ws);
    e = sort_and_segment(grad->row_idx, n, c, r, L, w, nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, d_err,
                         stream);
    if (e == cudaSuccess) e = fused_rows_sgd_sorted(w, L, grad->vals, c, P, vec4, d_err, stream);
    return from_cuda(e);
}

sparse_status_t sparse_sgd_step(float* p, float* buf, int64_t dim, const int64_t* idx, const float* g, int64_t nnz,
                                int is_canonical, sparse_sgd_config_t cfg, void* ws, size_t ws_bytes, int32_t* d_err,
                                cudaStream_t stream)
{
    sparse_grad_t grad{};
    grad.form = SPARSE_GRAD_ROW_COO;
    grad.n = nnz;
    grad.row_idx = idx;
    grad.vals = g;
    grad.is_canonical = is_canonical;
    return sparse_sgd_table_step(p, buf, dim, 1, &grad, cfg, ws, ws_bytes, d_err, stream);
}

sparse_status_t sparse_check_finite(const float* vals, int64_t n, int32_t* d_err, cudaStream_t stream)
{
    if (n < 0 || d_err == nullptr || (n > 0 && vals == nullptr)) return SPARSE_ERR_INVALID_ARG;
    return from_cuda(check_finite(vals, n, d_err, stream));
}

sparse_status_t sparse_check_state(const float* m, const float* v, int64_t r, int64_t c, const sparse_grad_t* grad,
                                   int32_t* d_err, cudaStream_t stream)
{
    sparse_status_t st = check_grad(grad, r, c);
    if (st) return st;
    if (d_err == nullptr || (r > 0 && (m == nullptr || v == nullptr))) return SPARSE_ERR_INVALID_ARG;
    const int64_t n = grad->n;
    if (grad->form == SPARSE_GRAD_CSR) {
        cudaError_t e = csr_check(grad->row_off, grad->cols, r, c, n, 0, nullptr, 0, 0, nullptr, nullptr, nullptr, d_err, stream);
        if (e == cudaSuccess && n > 0) e = check_state_csr(grad->row_off, grad->cols, r, c, n, m, v, d_err, stream);
        return from_cuda(e);
    }
    const int vec4 = (c % 4 == 0) && aligned16(m) && aligned16(v);
    return from_cuda(check_state_rows(m, v, r, c, grad->row_idx, n, vec4, d_err, stream));
}

sparse_status_t sparse_read_rows(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out,
                                 int32_t* d_err, cudaStream_t stream)
{
    if (r < 0 || c < 1 || n < 0 || d_err == nullptr) return SPARSE_ERR_INVALID_ARG;
    if (r > 0 && c > INT64_MAX / r) return SPARSE_ERR_INVALID_ARG;
    if (n == 0) return SPARSE_OK;
    if (idx == nullptr || out == nullptr || (r > 0 && table == nullptr)) return SPARSE_ERR_INVALID_ARG;
    const int vec4 = (c % 4 == 0) && aligned16(table) && aligned16(out);
    return from_cuda(read_rows(table, r, c, idx, n, out, vec4, d_err, stream));
}

}  // extern "C"
