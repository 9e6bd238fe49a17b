// gather.cu -- streaming passes over caller arrays outside the step proper: the
// finiteness check of gradient values and the check of the moment state a step
// would read ("DiskSparseAdam (DSA)" README, "Validated Inputs": non-finite
// gradients and NaN / negative moment rows are explicit errors), and the row
// gather.
//
// Row gather: out[i, :] = table[idx[i], :], the lookup that feeds the
// forward pass ("DiskSparseAdam (DSA)" README, API read_rows(indices): the rows
// of the table at the given indices, indices validated).
//
// A team of T lanes owns one output row at a time, each lane NV vectors of V
// floats (128-bit loads and stores when c % 4 == 0 and both arrays are 16-byte
// aligned); a team requests kGatherRows rows before storing any, and rows wider
// than T*NV*V columns are walked in chunks.  The copy is bit for bit.  A bad
// index sets SPARSE_ERR_INDEX_OUT_OF_RANGE and its output row is not written.
#include <algorithm>

#include "fused.cuh"
#include "profile.cuh"

namespace so {

constexpr int kGatherRows = 4;

template <int T, int NV, int V>
__global__ void __launch_bounds__(kBlock) k_read_rows(const float* __restrict__ table, int64_t r, int64_t c,
                                                      const int64_t* __restrict__ idx, int64_t n,
                                                      float* __restrict__ out, int32_t* d_err)
{
    pdl_wait();   // writes a caller output: dependents start after this grid exits
    constexpr int kTeams = kBlock / T;
    constexpr int CW = T * NV * V;
    constexpr int R = kGatherRows;
    const int lane = threadIdx.x & 31;
    const int tl = lane & (T - 1);
    const int64_t team_g = static_cast<int64_t>(blockIdx.x) * kTeams + threadIdx.x / T;
    const int64_t nteams = static_cast<int64_t>(gridDim.x) * kTeams;
    const int nchunks = static_cast<int>((c + CW - 1) / CW);
    for (int64_t i0 = team_g * R; i0 < n; i0 += nteams * R) {
        int64_t row[R];
        bool ok[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            row[u] = (i0 + u < n) ? idx[i0 + u] : -1;
            ok[u] = row[u] >= 0 && row[u] < r;
            if (i0 + u < n && !ok[u] && tl == 0) set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
        }
        for (int cc = 0; cc < nchunks; ++cc) {
            const int64_t col0 = static_cast<int64_t>(cc) * CW;
            float x[R][NV][V];
#pragma unroll
            for (int u = 0; u < R; ++u) {
                if (!ok[u]) continue;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) ld_state<V>(table + row[u] * c + col, x[u][k]);
                }
            }
#pragma unroll
            for (int u = 0; u < R; ++u) {
                if (!ok[u]) continue;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) st_state<V>(out + (i0 + u) * c + col, x[u][k]);
                }
            }
        }
    }
}

template <int T, int NV, int V>
static cudaError_t launch_gather(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out,
                                 int32_t* d_err, cudaStream_t s)
{
    constexpr int kTeams = kBlock / T;
    static const int occ = [] {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_read_rows<T, NV, V>, kBlock, 0);
        return o > 0 ? o : 1;
    }();
    const int64_t want = (n + static_cast<int64_t>(kTeams) * kGatherRows - 1) / (static_cast<int64_t>(kTeams) * kGatherRows);
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(occ) * num_sms())));
    SO_PROFILE("read_rows", s);
    launch(k_read_rows<T, NV, V>, dim3(blocks), dim3(kBlock), s, table, r, c, idx, n, out, d_err);
    return cudaGetLastError();
}

// Any NaN or infinity among n values sets SPARSE_ERR_NON_FINITE.  Grid-stride,
// 128-bit loads over the 16-byte aligned body, scalar head and tail.
__global__ void __launch_bounds__(kBlock) k_check_finite(const float* __restrict__ vals, int64_t n, int64_t head,
                                                         int32_t* d_err)
{
    pdl_enter();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    bool bad = false;
    for (int64_t i = tid; i < head && i < n; i += stride) bad |= !isfinite(vals[i]);
    const int64_t nv = (n - head) / 4;
    const float4* body = reinterpret_cast<const float4*>(vals + head);
    for (int64_t i = tid; i < nv; i += stride) {
        const float4 q = __ldcs(body + i);
        bad |= !isfinite(q.x) || !isfinite(q.y) || !isfinite(q.z) || !isfinite(q.w);
    }
    for (int64_t i = head + nv * 4 + tid; i < n; i += stride) bad |= !isfinite(vals[i]);
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(d_err, SPARSE_ERR_NON_FINITE);
}

// A moment value a step must not read: m not finite; v not finite or below zero
// (-0.0 is not below zero).
__device__ __forceinline__ bool bad_moments(float m, float v) { return !isfinite(m) || !isfinite(v) || v < 0.0f; }

// Moment state of the rows a row-COO gradient lists (repeats allowed, any
// order): every column of m and v of each listed row.  Teams and loads as in the
// row gather; a bad index sets SPARSE_ERR_INDEX_OUT_OF_RANGE and is skipped, a
// bad moment SPARSE_ERR_BAD_STATE.  Reads only; m and v are not streamed (the
// step that follows reads the same rows).
template <int T, int NV, int V>
__global__ void __launch_bounds__(kBlock) k_check_state_rows(const float* __restrict__ m, const float* __restrict__ v,
                                                             int64_t r, int64_t c, const int64_t* __restrict__ idx,
                                                             int64_t n, int32_t* d_err)
{
    pdl_enter();
    constexpr int kTeams = kBlock / T;
    constexpr int CW = T * NV * V;
    constexpr int R = kGatherRows;
    const int lane = threadIdx.x & 31;
    const int tl = lane & (T - 1);
    const int64_t team_g = static_cast<int64_t>(blockIdx.x) * kTeams + threadIdx.x / T;
    const int64_t nteams = static_cast<int64_t>(gridDim.x) * kTeams;
    const int nchunks = static_cast<int>((c + CW - 1) / CW);
    bool bad = false;
    for (int64_t i0 = team_g * R; i0 < n; i0 += nteams * R) {
        int64_t row[R];
        bool ok[R];
#pragma unroll
        for (int u = 0; u < R; ++u) {
            row[u] = (i0 + u < n) ? idx[i0 + u] : -1;
            ok[u] = row[u] >= 0 && row[u] < r;
            if (i0 + u < n && !ok[u] && tl == 0) set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
        }
        for (int cc = 0; cc < nchunks; ++cc) {
            const int64_t col0 = static_cast<int64_t>(cc) * CW;
            float xm[R][NV][V], xv[R][NV][V];
#pragma unroll
            for (int u = 0; u < R; ++u) {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (ok[u] && col < c) {
                        ld_state<V>(m + row[u] * c + col, xm[u][k]);
                        ld_state<V>(v + row[u] * c + col, xv[u][k]);
                    } else {
#pragma unroll
                        for (int e = 0; e < V; ++e) xm[u][k][e] = xv[u][k][e] = 0.0f;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < R; ++u)
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int e = 0; e < V; ++e) bad |= bad_moments(xm[u][k][e], xv[u][k][e]);
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(d_err, SPARSE_ERR_BAD_STATE);
}

template <int T, int NV, int V>
static cudaError_t launch_check_state(const float* m, const float* v, int64_t r, int64_t c, const int64_t* idx,
                                     int64_t n, int32_t* d_err, cudaStream_t s)
{
    constexpr int kTeams = kBlock / T;
    static const int occ = [] {
        int o = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_check_state_rows<T, NV, V>, kBlock, 0);
        return o > 0 ? o : 1;
    }();
    const int64_t want = (n + static_cast<int64_t>(kTeams) * kGatherRows - 1) / (static_cast<int64_t>(kTeams) * kGatherRows);
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(occ) * num_sms())));
    SO_PROFILE("check_state_rows", s);
    launch(k_check_state_rows<T, NV, V>, dim3(blocks), dim3(kBlock), s, m, v, r, c, idx, n, d_err);
    return cudaGetLastError();
}

cudaError_t check_state_rows(const float* m, const float* v, int64_t r, int64_t c, const int64_t* idx, int64_t n,
                             int vec4, int32_t* d_err, cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    if (vec4) {
        const int64_t nv = c / 4;
        if (nv <= 1) return launch_check_state<1, 1, 4>(m, v, r, c, idx, n, d_err, s);
        if (nv <= 2) return launch_check_state<2, 1, 4>(m, v, r, c, idx, n, d_err, s);
        if (nv <= 4) return launch_check_state<4, 1, 4>(m, v, r, c, idx, n, d_err, s);
        if (nv <= 8) return launch_check_state<8, 1, 4>(m, v, r, c, idx, n, d_err, s);
        if (nv <= 16) return launch_check_state<16, 1, 4>(m, v, r, c, idx, n, d_err, s);
        if (nv <= 32) return launch_check_state<32, 1, 4>(m, v, r, c, idx, n, d_err, s);
        return launch_check_state<32, 2, 4>(m, v, r, c, idx, n, d_err, s);
    }
    if (c <= 1) return launch_check_state<1, 1, 1>(m, v, r, c, idx, n, d_err, s);
    if (c <= 2) return launch_check_state<2, 1, 1>(m, v, r, c, idx, n, d_err, s);
    if (c <= 4) return launch_check_state<4, 1, 1>(m, v, r, c, idx, n, d_err, s);
    if (c <= 8) return launch_check_state<8, 1, 1>(m, v, r, c, idx, n, d_err, s);
    if (c <= 16) return launch_check_state<16, 1, 1>(m, v, r, c, idx, n, d_err, s);
    if (c <= 32) return launch_check_state<32, 1, 1>(m, v, r, c, idx, n, d_err, s);
    return launch_check_state<32, 4, 1>(m, v, r, c, idx, n, d_err, s);
}

cudaError_t check_finite(const float* vals, int64_t n, int32_t* d_err, cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    const int64_t mis = static_cast<int64_t>((reinterpret_cast<uintptr_t>(vals) & 15u) / 4);
    const int64_t head = mis ? std::min<int64_t>(4 - mis, n) : 0;
    const int64_t want = (n / 4 + kBlock - 1) / kBlock + 1;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8 * num_sms())));
    SO_PROFILE("check_finite", s);
    launch(k_check_finite, dim3(blocks), dim3(kBlock), s, vals, n, head, d_err);
    return cudaGetLastError();
}

cudaError_t read_rows(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out, int vec4,
                      int32_t* d_err, cudaStream_t s)
{
    if (n <= 0) return cudaSuccess;
    if (vec4) {
        const int64_t nv = c / 4;
        if (nv <= 1) return launch_gather<1, 1, 4>(table, r, c, idx, n, out, d_err, s);
        if (nv <= 2) return launch_gather<2, 1, 4>(table, r, c, idx, n, out, d_err, s);
        if (nv <= 4) return launch_gather<4, 1, 4>(table, r, c, idx, n, out, d_err, s);
        if (nv <= 8) return launch_gather<8, 1, 4>(table, r, c, idx, n, out, d_err, s);
        if (nv <= 16) return launch_gather<16, 1, 4>(table, r, c, idx, n, out, d_err, s);
        if (nv <= 32) return launch_gather<32, 1, 4>(table, r, c, idx, n, out, d_err, s);
        return launch_gather<32, 2, 4>(table, r, c, idx, n, out, d_err, s);
    }
    if (c <= 1) return launch_gather<1, 1, 1>(table, r, c, idx, n, out, d_err, s);
    if (c <= 2) return launch_gather<2, 1, 1>(table, r, c, idx, n, out, d_err, s);
    if (c <= 4) return launch_gather<4, 1, 1>(table, r, c, idx, n, out, d_err, s);
    if (c <= 8) return launch_gather<8, 1, 1>(table, r, c, idx, n, out, d_err, s);
    if (c <= 16) return launch_gather<16, 1, 1>(table, r, c, idx, n, out, d_err, s);
    if (c <= 32) return launch_gather<32, 1, 1>(table, r, c, idx, n, out, d_err, s);
    return launch_gather<32, 4, 1>(table, r, c, idx, n, out, d_err, s);
}

}  // namespace so
