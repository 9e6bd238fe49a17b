// csr.cu -- element-granular CSR gradients and the CSR <-> COO conversions.
// "Module sparse_optimizer" (optirs-gpu 0.3.2 docs), "Sparse gradient
// representations": CSR row_offsets / col_indices (strictly ascending within a
// row) / values with the dense shape; CsrGradient::to_coo / from_coo by the
// linear index row*c + col.
//
// Row traversal: one warp per group of 32 consecutive rows.  Lane l loads
// row_off[r0 + l] (coalesced); the group's entries are the contiguous range
// row_off[r0] .. row_off[r0 + 32], walked 32 at a time, and the row of entry j
// is the last lane whose row start is <= j (a 5-step shuffle search).  Empty
// rows cost one coalesced offset load each.
#include <algorithm>

#include "fused.cuh"
#include "profile.cuh"

namespace so {

constexpr int kMergeItems = 16;

struct Group {
    int64_t a, b;    // this lane's row: entries [a, b)
    int64_t lo, hi;  // the group's entries
    bool ok;         // offsets of the group well formed
};

__device__ __forceinline__ Group load_group(const int64_t* __restrict__ row_off, int64_t r, int64_t nnz,
                                            int64_t r0, int lane)
{
    Group G;
    const int64_t rr = r0 + lane;
    G.a = row_off[rr < r ? rr : r];
    const int64_t last = row_off[(r0 + 32) < r ? (r0 + 32) : r];
    G.b = __shfl_down_sync(kFull, G.a, 1);
    if (lane == 31) G.b = last;
    G.lo = __shfl_sync(kFull, G.a, 0);
    G.hi = last;
    const bool mine = (rr >= r) || (G.a >= 0 && G.a <= G.b && G.b <= nnz);
    G.ok = __all_sync(kFull, mine);
    return G;
}

// Lane whose row holds entry j: the largest l with row start a_l <= j.  Every
// lane of the warp must call (shuffles); src lanes stay within 0..31.
__device__ __forceinline__ int row_lane(const Group& G, int64_t j)
{
    int l = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) {
        const int64_t ac = __shfl_sync(kFull, G.a, l + step);
        if (ac <= j) l += step;
    }
    return l;
}

// Validation of a CSR gradient (and of last_step < t on its touched coordinates).
__global__ void __launch_bounds__(kBlock) k_csr_check(const int64_t* __restrict__ row_off,
                                                      const int32_t* __restrict__ cols, int64_t r,
                                                      int64_t c, int64_t nnz, int full_rows,
                                                      const int64_t* __restrict__ ls, int ls_per_coord,
                                                      int64_t t, int32_t* d_err)
{
    pdl_enter();
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0 && (row_off[0] != 0 || row_off[r] != nnz))
        set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32; gi < groups;
         gi += gstride) {
        const int64_t r0 = gi * 32;
        const Group G = load_group(row_off, r, nnz, r0, lane);
        if (!G.ok) {
            if (lane == 0) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
            continue;
        }
        const int64_t rr = r0 + lane;
        if (rr < r && G.b > G.a) {
            if (full_rows && G.b - G.a != c) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
            if (ls && !ls_per_coord && ls[rr] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
        }
        for (int64_t base = G.lo; base < G.hi; base += 32) {
            const int64_t j = base + lane;
            const int l = row_lane(G, j);
            const int64_t start = __shfl_sync(kFull, G.a, l);
            if (j >= G.hi) continue;
            const int32_t col = cols[j];
            if (col < 0 || col >= c) {
                set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
                continue;
            }
            if (j > start && cols[j - 1] >= col) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
            if (ls && ls_per_coord && ls[(r0 + l) * c + col] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
        }
    }
}

// Element-granular update: every listed coordinate independently.  A per-row
// last_step is read by every coordinate of the row and written once per row
// after the whole group has read it.
template <class Op>
__global__ void __launch_bounds__(kBlock) k_csr_update(const int64_t* __restrict__ row_off,
                                                       const int32_t* __restrict__ cols,
                                                       const float* __restrict__ vals, int64_t r, int64_t c,
                                                       int64_t nnz, Op op, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int lane = threadIdx.x & 31;
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32; gi < groups;
         gi += gstride) {
        const int64_t r0 = gi * 32;
        const Group G = load_group(row_off, r, nnz, r0, lane);
        if (!G.ok) continue;
        for (int64_t base = G.lo; base < G.hi; base += 32) {
            const int64_t j = base + lane;
            const int l = row_lane(G, j);
            if (j >= G.hi) continue;
            op.coord(r0 + l, static_cast<int64_t>(__ldcs(cols + j)), __ldcs(vals + j));
        }
        __syncwarp();
        const int64_t rr = r0 + lane;
        if (rr < r && G.b > G.a) op.row_done(rr);
    }
}

struct CsrAdamOp {
    AdamParams P;
    int64_t c;
    __device__ __forceinline__ void coord(int64_t row, int64_t col, float g) const
    {
        const int64_t i = row * c + col;
        float b1 = P.beta1, b2 = P.beta2;
        if (P.dd) dormancy_factors(P, P.t - P.ls[P.ls_per_coord ? i : row], b1, b2);
        float p = P.p[i], m = P.m[i], v = P.v[i];
        adam_coord(P, b1, b2, g, p, m, v);
        P.p[i] = p;
        P.m[i] = m;
        P.v[i] = v;
        if (P.ls_per_coord) P.ls[i] = P.t;
    }
    __device__ __forceinline__ void row_done(int64_t row) const
    {
        if (!P.ls_per_coord) P.ls[row] = P.t;
    }
};

struct CsrSgdOp {
    SgdParams P;
    int64_t c;
    __device__ __forceinline__ void coord(int64_t row, int64_t col, float g) const
    {
        const int64_t i = row * c + col;
        float p = P.p[i];
        float b = P.buf ? P.buf[i] : 0.0f;
        sgd_coord(P, g, p, b);
        P.p[i] = p;
        if (P.buf) P.buf[i] = b;
    }
    __device__ __forceinline__ void row_done(int64_t) const {}
};

static int group_blocks(int64_t r)
{
    const int64_t groups = (r + 31) / 32;
    const int64_t want = (groups + kBlock / 32 - 1) / (kBlock / 32);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 16 * num_sms())));
}

cudaError_t csr_check(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                      int full_rows, const int64_t* ls, int ls_per_coord, int64_t t, int32_t* d_err,
                      cudaStream_t s)
{
    SO_PROFILE("csr_check", s);
    launch(k_csr_check, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, r, c, nnz, full_rows, ls, ls_per_coord, t,
                                                   d_err);
    return cudaGetLastError();
}

cudaError_t csr_adam(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r, int64_t c,
                     int64_t nnz, const AdamParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_update_adam", s);
    launch(k_csr_update<CsrAdamOp>, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, vals, r, c, nnz,
                                                               CsrAdamOp{P, c}, d_err);
    return cudaGetLastError();
}

cudaError_t csr_sgd(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r, int64_t c,
                    int64_t nnz, const SgdParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_update_sgd", s);
    launch(k_csr_update<CsrSgdOp>, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, vals, r, c, nnz,
                                                              CsrSgdOp{P, c}, d_err);
    return cudaGetLastError();
}

// CsrGradient::to_coo: lin[j] = row(j)*c + cols[j].
__global__ void __launch_bounds__(kBlock) k_csr_to_coo(const int64_t* __restrict__ row_off,
                                                       const int32_t* __restrict__ cols, int64_t r, int64_t c,
                                                       int64_t nnz, int64_t* __restrict__ lin, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int lane = threadIdx.x & 31;
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32; gi < groups;
         gi += gstride) {
        const int64_t r0 = gi * 32;
        const Group G = load_group(row_off, r, nnz, r0, lane);
        if (!G.ok) continue;
        for (int64_t base = G.lo; base < G.hi; base += 32) {
            const int64_t j = base + lane;
            const int l = row_lane(G, j);
            if (j < G.hi) lin[j] = (r0 + l) * c + static_cast<int64_t>(cols[j]);
        }
    }
}

cudaError_t csr_to_coo(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                       int64_t* lin_out, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_to_coo", s);
    launch(k_csr_to_coo, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, r, c, nnz, lin_out, d_err);
    return cudaGetLastError();
}

// Sorted keys strictly ascending and in [0, bound).
__global__ void __launch_bounds__(kBlock) k_check_ascending(const int64_t* __restrict__ keys, int64_t n,
                                                            int64_t bound, int32_t* d_err)
{
    pdl_enter();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride) {
        const int64_t k = keys[i];
        if (k < 0 || k >= bound)
            set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
        else if (i > 0 && keys[i - 1] >= k)
            set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
    }
}

// Merge path of A = {i*scale : i = 0..r} with sorted B = keys[0..nb), A first on
// ties.  Taking A[i] with j entries of B already taken gives row_off[i] = j*mult
// (the number of keys below row i's first linear index).  Taking B[j] (only when
// cols != nullptr) writes its column keys[j] - (i-1)*scale.  Each thread merges
// kMergeItems consecutive elements after a binary search of its diagonal.
__global__ void __launch_bounds__(kBlock) k_merge_offsets(const int64_t* __restrict__ keys, int64_t nb,
                                                          int64_t r, int64_t scale, int64_t mult,
                                                          int64_t* __restrict__ row_off,
                                                          int32_t* __restrict__ cols, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int64_t total = r + 1 + nb;
    const int64_t d0 = (static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x) * kMergeItems;
    if (d0 >= total) return;
    int64_t lo = d0 - nb > 0 ? d0 - nb : 0;
    int64_t hi = d0 < r + 1 ? d0 : r + 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (mid * scale <= keys[d0 - mid - 1])
            lo = mid + 1;
        else
            hi = mid;
    }
    int64_t i = lo, j = d0 - lo;
    for (int k = 0; k < kMergeItems && i + j < total; ++k) {
        if (i <= r && (j >= nb || i * scale <= keys[j])) {
            row_off[i] = j * mult;
            ++i;
        } else {
            if (cols) cols[j] = static_cast<int32_t>(keys[j] - (i - 1) * scale);
            ++j;
        }
    }
}

__global__ void __launch_bounds__(kBlock) k_fill_cols(int32_t* __restrict__ cols, int64_t total, int64_t c,
                                                      int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; e < total; e += stride)
        cols[e] = static_cast<int32_t>(e % c);
}

static int flat_blocks(int64_t n, int64_t per_thread)
{
    const int64_t want = (n + kBlock * per_thread - 1) / (kBlock * per_thread);
    return static_cast<int>(std::max<int64_t>(1, want));
}

cudaError_t coo_to_csr(const int64_t* lin, int64_t nnz, int64_t r, int64_t c, int64_t* row_off_out,
                       int32_t* cols_out, int32_t* d_err, cudaStream_t s)
{
    if (nnz > 0) {
        const int blocks = static_cast<int>(std::min<int64_t>(flat_blocks(nnz, 1), 8 * num_sms()));
        SO_PROFILE("check_ascending", s);
        launch(k_check_ascending, dim3(blocks), dim3(kBlock), s, lin, nnz, r * c, d_err);
    }
    SO_PROFILE("merge_offsets", s);
    launch(k_merge_offsets, dim3(flat_blocks(r + 1 + nnz, kMergeItems)), dim3(kBlock), s, lin, nnz, r, c, 1,
           row_off_out, cols_out, d_err);
    return cudaGetLastError();
}

cudaError_t row_coo_to_csr(const int64_t* rows, int64_t nrows, int64_t r, int64_t c, int64_t* row_off_out,
                           int32_t* cols_out, int32_t* d_err, cudaStream_t s)
{
    if (nrows > 0) {
        const int blocks = static_cast<int>(std::min<int64_t>(flat_blocks(nrows, 1), 8 * num_sms()));
        SO_PROFILE("check_ascending", s);
        launch(k_check_ascending, dim3(blocks), dim3(kBlock), s, rows, nrows, r, d_err);
    }
    {
        SO_PROFILE("merge_offsets", s);
        launch(k_merge_offsets, dim3(flat_blocks(r + 1 + nrows, kMergeItems)), dim3(kBlock), s, rows, nrows, r,
               1, c, row_off_out, nullptr, d_err);
    }
    if (nrows > 0) {
        SO_PROFILE("fill_cols", s);
        const int blocks = static_cast<int>(std::min<int64_t>(flat_blocks(nrows * c, 4), 16 * num_sms()));
        launch(k_fill_cols, dim3(blocks), dim3(kBlock), s, cols_out, nrows * c, c, d_err);
    }
    return cudaGetLastError();
}

}  // namespace so
