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
// Batches of full rows a warp requests at once in the check and in the update.
#ifndef SO_CSR_CHECK_ILP
#define SO_CSR_CHECK_ILP 4
#endif
#ifndef SO_CSR_ROW_ILP
#define SO_CSR_ROW_ILP 2
#endif
constexpr int kCsrCheckIlp = SO_CSR_CHECK_ILP;
constexpr int kCsrRowIlp = SO_CSR_ROW_ILP;

struct Group {
    int64_t a, b;    // this lane's row: entries [a, b)
    int64_t lo, hi;  // the group's entries
    bool ok;         // offsets of the group well formed
};

// The two offsets a lane needs for the group at r0 (requested ahead of use).
struct GroupRaw {
    int64_t a, last;
};
__device__ __forceinline__ GroupRaw fetch_group(const int64_t* __restrict__ row_off, int64_t r, int64_t r0, int lane)
{
    GroupRaw g{0, 0};
    if (r0 < r) {
        const int64_t rr = r0 + lane;
        g.a = row_off[rr < r ? rr : r];
        g.last = row_off[(r0 + 32) < r ? (r0 + 32) : r];
    }
    return g;
}

__device__ __forceinline__ Group make_group(const GroupRaw& raw, int64_t r, int64_t nnz, int64_t r0, int lane);
__device__ __forceinline__ Group load_group(const int64_t* __restrict__ row_off, int64_t r, int64_t nnz,
                                            int64_t r0, int lane)
{
    return make_group(fetch_group(row_off, r, r0, lane), r, nnz, r0, lane);
}

__device__ __forceinline__ Group make_group(const GroupRaw& raw, int64_t r, int64_t nnz, int64_t r0, int lane)
{
    Group G;
    const int64_t rr = r0 + lane;
    G.a = raw.a;
    const int64_t last = raw.last;
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

// Full rows (all c columns listed, c = 4*TQ <= 128) are handled by sub-teams of
// TQ lanes, one float4 of the row per lane, 32/TQ rows at a time and two such
// batches requested together; the entries of the other rows are walked 32 at a
// time, two chunks requested together, skipping the full rows.  fullmask has
// bit l set when the group's row r0 + l is a full row taking that path.
template <int TQ>
__device__ __forceinline__ unsigned full_row_mask(const Group& G, int64_t r0, int64_t r, int64_t c)
{
    if constexpr (TQ == 0) {
        return 0u;
    } else {
        const int64_t rr = r0 + (threadIdx.x & 31);
        return __ballot_sync(kFull, rr < r && G.b - G.a == c && (G.a & 3) == 0);
    }
}

// Lane l of the warp's k-th full row (k < popc(mask)).
__device__ __forceinline__ int nth_row(unsigned mask, int k) { return static_cast<int>(__fns(mask, 0, k + 1)); }

// Validation of a CSR gradient whose rows need not be full (and of last_step < t
// on its touched coordinates).  With ent_row: every entry's row, and with ent_gap
// its t - last_step (per-coordinate last_step; at most INT32_MAX), for the flat
// update.
template <int TQ>
__global__ void __launch_bounds__(kBlock) k_csr_check(const int64_t* __restrict__ row_off,
                                                      const int32_t* __restrict__ cols, int64_t r,
                                                      int64_t c, int64_t nnz,
                                                      const int64_t* __restrict__ ls, int ls_per_coord,
                                                      int64_t t, int32_t* __restrict__ ent_row,
                                                      int32_t* __restrict__ ent_gap, int32_t* d_err)
{
    const auto gap_of = [t](int64_t last) {
        const int64_t gap = t - last;
        return static_cast<int32_t>(gap < INT32_MAX ? gap : INT32_MAX);
    };
    pdl_enter();
    const int lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && threadIdx.x == 0 && (row_off[0] != 0 || row_off[r] != nnz))
        set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32;
    GroupRaw next = fetch_group(row_off, r, gi * 32, lane);
    for (; gi < groups; gi += gstride) {
        const int64_t r0 = gi * 32;
        const GroupRaw cur = next;
        next = fetch_group(row_off, r, (gi + gstride) * 32, lane);   // the next group's offsets, in flight
        const Group G = make_group(cur, r, nnz, r0, lane);
        if (!G.ok) {
            if (lane == 0) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
            continue;
        }
        const int64_t rr = r0 + lane;
        if (rr < r && G.b > G.a && ls && !ls_per_coord && ls[rr] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
        const unsigned fullmask = full_row_mask<TQ>(G, r0, r, c);
        if constexpr (TQ > 0) {
            // a listed full row is canonical iff its columns are exactly 0 .. c-1
            constexpr int RPI = 32 / TQ;
            const int sub = lane / TQ, q = lane % TQ;
            const int nfull = __popc(fullmask);
            constexpr int U = kCsrCheckIlp;   // batches of rows whose columns are requested together
            for (int k0 = 0; k0 < nfull; k0 += U * RPI) {
                int4 cc[U];
                int lr[U];
                bool act[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * RPI + sub;
                    act[u] = k < nfull;
                    lr[u] = act[u] ? nth_row(fullmask, k) : 0;
                    const int64_t a = __shfl_sync(kFull, G.a, lr[u]);
                    if (act[u]) cc[u] = *reinterpret_cast<const int4*>(cols + a + 4 * q);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!act[u]) continue;
                    const int want = 4 * q;
                    if (cc[u].x != want || cc[u].y != want + 1 || cc[u].z != want + 2 || cc[u].w != want + 3) {
                        const bool out = cc[u].x < 0 || cc[u].x >= c || cc[u].y < 0 || cc[u].y >= c ||
                                         cc[u].z < 0 || cc[u].z >= c || cc[u].w < 0 || cc[u].w >= c;
                        set_error(d_err, out ? SPARSE_ERR_INDEX_OUT_OF_RANGE : SPARSE_ERR_NOT_CANONICAL);
                    }
                    const int64_t a = __shfl_sync(kFull, G.a, lr[u]) + 4 * q;   // this lane's four entries
                    if (ls && ls_per_coord) {
                        const int64_t i = (r0 + lr[u]) * c + 4 * q;
                        for (int e = 0; e < 4; ++e) {
                            const int64_t last = ls[i + e];
                            if (last >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
                            if (ent_gap) ent_gap[a + e] = gap_of(last);
                        }
                    }
                    if (ent_row) {
                        for (int e = 0; e < 4; ++e) ent_row[a + e] = static_cast<int32_t>(r0 + lr[u]);
                    }
                }
            }
        }
        for (int64_t base = G.lo; base < G.hi; base += 64) {
            int64_t j[2];
            int l[2];
            bool act[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                j[u] = base + 32 * u + lane;
                l[u] = row_lane(G, j[u]);
                act[u] = j[u] < G.hi && !((fullmask >> l[u]) & 1u);
            }
            if (!__any_sync(kFull, act[0] || act[1])) continue;
            int32_t col[2], prev[2];
            int64_t start[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                start[u] = __shfl_sync(kFull, G.a, l[u]);
                col[u] = act[u] ? cols[j[u]] : 0;
                prev[u] = (act[u] && j[u] > start[u]) ? cols[j[u] - 1] : -1;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (!act[u]) continue;
                if (col[u] < 0 || col[u] >= c) {
                    set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
                    continue;
                }
                if (prev[u] >= col[u]) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
                if (ls && ls_per_coord) {
                    const int64_t last = ls[(r0 + l[u]) * c + col[u]];
                    if (last >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
                    if (ent_gap) ent_gap[j[u]] = gap_of(last);
                }
                if (ent_row) ent_row[j[u]] = static_cast<int32_t>(r0 + l[u]);
            }
        }
    }
}

// Validation when every listed row must be full (per-row last_step): thread i
// takes rows i, i + stride, ... kFullRowIlp at a time, all their offsets
// requested together (one coalesced pair of loads per warp and row batch); a
// non-empty row must hold exactly c entries (its start then a multiple of c,
// the offsets starting at 0), is recorded as rows_list[start / c] and has its
// last_step checked.  Each row's own offsets are checked to lie in [0, nnz) in
// order before its slot is written, so a malformed CSR never writes outside
// rows_list[0 .. nnz/c).  Then one flat pass over the column array: entry j must
// be column j % c (four entries a thread at a time where the array is aligned).
// The CSR is the call's input, so the first batch of offsets and the column pass
// are read and checked before the wait for the previous kernel on the stream; the
// problems found are only recorded then and written to *d_err after the wait (a
// previous kernel may still read the error word), as are rows_list (workspace
// the previous kernel may use) and the last_step checks (last_step it may write).
constexpr int kFullRowIlp = 4;
__global__ void __launch_bounds__(kBlock) k_csr_check_full(const int64_t* __restrict__ row_off,
                                                           const int32_t* __restrict__ cols, int64_t r, int64_t c,
                                                           int64_t nnz, const int64_t* __restrict__ ls, int64_t t,
                                                           int64_t* __restrict__ rows_list, int32_t* d_err)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x;
    int bad = 0;   // SPARSE_ERR_NOT_CANONICAL or SPARSE_ERR_INDEX_OUT_OF_RANGE found before the wait
    if (i0 == 0 && (row_off[0] != 0 || row_off[r] != nnz)) bad = SPARSE_ERR_NOT_CANONICAL;
    const auto load = [&](int64_t base, int64_t (&a)[kFullRowIlp], int64_t (&b)[kFullRowIlp]) {
#pragma unroll
        for (int u = 0; u < kFullRowIlp; ++u) {
            const int64_t rr = base + u * stride;
            a[u] = rr < r ? row_off[rr] : 0;
            b[u] = rr < r ? row_off[rr + 1] : 0;
        }
    };
    // a row is taken (listed and checked) when its offsets are well formed
    const auto well_formed = [&](int64_t a, int64_t b) {
        return a >= 0 && a <= b && b <= nnz && b - a == c && a % c == 0;
    };
    int64_t a0[kFullRowIlp], b0[kFullRowIlp];
    load(i0, a0, b0);
#pragma unroll
    for (int u = 0; u < kFullRowIlp; ++u)
        if (i0 + u * stride < r && a0[u] != b0[u] && !well_formed(a0[u], b0[u])) bad = SPARSE_ERR_NOT_CANONICAL;
    const bool vec = (reinterpret_cast<uintptr_t>(cols) & 15u) == 0;
    const int64_t n4 = vec ? nnz / 4 : 0;
    for (int64_t q = i0; q < n4; q += stride) {
        const int4 v = *reinterpret_cast<const int4*>(cols + 4 * q);
        const int32_t w[4] = {v.x, v.y, v.z, v.w};
        int64_t want = (4 * q) % c;   // column of entry 4q, then stepped with wrap-around
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (w[e] != want) bad = (w[e] < 0 || w[e] >= c) ? SPARSE_ERR_INDEX_OUT_OF_RANGE : SPARSE_ERR_NOT_CANONICAL;
            if (++want == c) want = 0;
        }
    }
    for (int64_t j = 4 * n4 + i0; j < nnz; j += stride) {
        const int32_t col = cols[j];
        if (col != j % c) bad = (col < 0 || col >= c) ? SPARSE_ERR_INDEX_OUT_OF_RANGE : SPARSE_ERR_NOT_CANONICAL;
    }
    pdl_enter();
    if (bad) set_error(d_err, bad);
    const auto take = [&](int64_t base, const int64_t (&a)[kFullRowIlp], const int64_t (&b)[kFullRowIlp]) {
#pragma unroll
        for (int u = 0; u < kFullRowIlp; ++u) {
            const int64_t rr = base + u * stride;
            if (rr >= r || a[u] == b[u] || !well_formed(a[u], b[u])) continue;
            if (rows_list) rows_list[a[u] / c] = rr;
            if (ls && ls[rr] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
        }
    };
    take(i0, a0, b0);
    for (int64_t base = i0 + stride * kFullRowIlp; base < r; base += stride * kFullRowIlp) {
        int64_t a[kFullRowIlp], b[kFullRowIlp];
        load(base, a, b);
#pragma unroll
        for (int u = 0; u < kFullRowIlp; ++u)
            if (base + u * stride < r && a[u] != b[u] && !well_formed(a[u], b[u])) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
        take(base, a, b);
    }
}

// Update.  Full rows go through the row epilogue of the fused kernels (128-bit
// state and gradient loads); the other entries are updated one coordinate per
// lane.  A per-row last_step is read by every coordinate of the row and written
// once per row after the whole group has read it.
template <class Op, class Epi, int TQ>
__global__ void __launch_bounds__(kBlock) k_csr_update(const int64_t* __restrict__ row_off,
                                                       const int32_t* __restrict__ cols,
                                                       const float* __restrict__ vals, int64_t r, int64_t c,
                                                       int64_t nnz, Op op, Epi epi, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int lane = threadIdx.x & 31;
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32;
    GroupRaw next = fetch_group(row_off, r, gi * 32, lane);
    for (; gi < groups; gi += gstride) {
        const int64_t r0 = gi * 32;
        const GroupRaw cur = next;
        next = fetch_group(row_off, r, (gi + gstride) * 32, lane);   // the next group's offsets, in flight
        const Group G = make_group(cur, r, nnz, r0, lane);
        if (!G.ok) continue;
        const unsigned fullmask = full_row_mask<TQ>(G, r0, r, c);
        if constexpr (TQ > 0) {
            constexpr int RPI = 32 / TQ;
            constexpr int A = Epi::kArrays;
            const int sub = lane / TQ, q = lane % TQ;
            const unsigned tmask = (TQ == 32) ? kFull : (((1u << TQ) - 1u) << (sub * TQ));
            const int nfull = __popc(fullmask);
            constexpr int U = kCsrRowIlp;   // batches of rows requested together
            for (int k0 = 0; k0 < nfull; k0 += U * RPI) {
                float x[U][A][4], g[U][4];
                int64_t row[U], last[U];
                bool act[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = k0 + u * RPI + sub;
                    act[u] = k < nfull;
                    const int l = act[u] ? nth_row(fullmask, k) : 0;
                    const int64_t a = __shfl_sync(kFull, G.a, l);
                    row[u] = r0 + l;
                    last[u] = 0;
                    if (act[u]) {
                        const int64_t off = row[u] * c + 4 * q;
#pragma unroll
                        for (int ar = 0; ar < A; ++ar)
                            if (ar < epi.arrays()) ld_state<4>(epi.array(ar) + off, x[u][ar]);
                        ld_grad<4>(vals + a + 4 * q, g[u]);
                        const int64_t* lp = op.row_last(row[u]);
                        if (lp) last[u] = *lp;
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (act[u]) {
                        const typename Epi::Row rw = op.make_row(row[u], last[u]);
                        epi.template apply<4>(rw, 4 * q, x[u], g[u]);
                        epi.end_row(rw, q, tmask);
                    }
                }
            }
        }
        for (int64_t base = G.lo; base < G.hi; base += 64) {
            int64_t j[2];
            int l[2];
            bool act[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                j[u] = base + 32 * u + lane;
                l[u] = row_lane(G, j[u]);
                act[u] = j[u] < G.hi && !((fullmask >> l[u]) & 1u);
            }
            if (!__any_sync(kFull, act[0] || act[1])) continue;
            int64_t col[2];
            float g[2];
            typename Op::Ld L[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                col[u] = act[u] ? static_cast<int64_t>(__ldcs(cols + j[u])) : 0;
                g[u] = act[u] ? __ldcs(vals + j[u]) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (act[u]) L[u] = op.load(r0 + l[u], col[u]);
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (act[u]) op.store(r0 + l[u], col[u], L[u], g[u]);
        }
        __syncwarp();
        const int64_t rr = r0 + lane;
        if (rr < r && G.b > G.a && !((fullmask >> lane) & 1u)) op.row_done(rr);
    }
}

struct CsrAdamOp {
    AdamParams P;
    int64_t c;
    struct Ld {
        float p, m, v;
        int64_t last;
    };
    __device__ __forceinline__ Ld load(int64_t row, int64_t col) const
    {
        const int64_t i = row * c + col;
        Ld L;
        L.p = P.p[i];
        L.m = P.m[i];
        L.v = P.v[i];
        L.last = P.dd ? P.ls[P.ls_per_coord ? i : row] : 0;
        return L;
    }
    __device__ __forceinline__ void store(int64_t row, int64_t col, Ld L, float g) const
    {
        const int64_t i = row * c + col;
        float b1 = P.beta1, b2 = P.beta2;
        if (P.dd) dormancy_factors(P, P.t - L.last, b1, b2);
        adam_coord(P, b1, b2, g, L.p, L.m, L.v);
        P.p[i] = L.p;
        P.m[i] = L.m;
        P.v[i] = L.v;
        if (P.ls_per_coord) P.ls[i] = P.t;
    }
    __device__ __forceinline__ void row_done(int64_t row) const
    {
        if (!P.ls_per_coord) P.ls[row] = P.t;
    }
    // full-row path: the per-row last_step the epilogue needs (DormancyDecay, per-row layout)
    __device__ __forceinline__ const int64_t* row_last(int64_t row) const
    {
        return (P.dd && !P.ls_per_coord) ? P.ls + row : nullptr;
    }
    __device__ __forceinline__ AdamEpi::Row make_row(int64_t row, int64_t last) const { return AdamEpi::Row{row, last}; }
};

struct CsrSgdOp {
    SgdParams P;
    int64_t c;
    struct Ld {
        float p, b;
    };
    __device__ __forceinline__ Ld load(int64_t row, int64_t col) const
    {
        const int64_t i = row * c + col;
        Ld L;
        L.p = P.p[i];
        L.b = P.buf ? P.buf[i] : 0.0f;
        return L;
    }
    __device__ __forceinline__ void store(int64_t row, int64_t col, Ld L, float g) const
    {
        const int64_t i = row * c + col;
        sgd_coord(P, g, L.p, L.b);
        P.p[i] = L.p;
        if (P.buf) P.buf[i] = L.b;
    }
    __device__ __forceinline__ void row_done(int64_t) const {}
    __device__ __forceinline__ const int64_t* row_last(int64_t) const { return nullptr; }
    __device__ __forceinline__ SgdEpi::Row make_row(int64_t row, int64_t) const { return SgdEpi::Row{row}; }
};

#ifndef SO_CSR_BLOCKS_PER_SM
#define SO_CSR_BLOCKS_PER_SM 16
#endif
// Blocks of the CSR kernels: one warp per group of 32 rows, at most
// SO_CSR_BLOCKS_PER_SM blocks per SM (several waves: a block that finds only
// empty groups retires quickly and its slot takes the next block).
// The check kernel's cap.
#ifndef SO_CSR_CHECK_BLOCKS_PER_SM
#define SO_CSR_CHECK_BLOCKS_PER_SM SO_CSR_BLOCKS_PER_SM
#endif
// Blocks per SM of the full-row check (one row per thread and pass).
#ifndef SO_CSR_FULL_BLOCKS_PER_SM
#define SO_CSR_FULL_BLOCKS_PER_SM 8
#endif
static int group_blocks(int64_t r, int per_sm = SO_CSR_BLOCKS_PER_SM)
{
    const int64_t groups = (r + 31) / 32;
    const int64_t want = (groups + kBlock / 32 - 1) / (kBlock / 32);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(per_sm) * num_sms())));
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sub-team size for full rows of c columns (one float4 per lane), or 0 when the
// rows take the per-coordinate path only.
static int full_row_team(int64_t c, bool aligned)
{
    if (!aligned || c % 4 != 0 || c > 128) return 0;
    const int64_t q = c / 4;
    return (q & (q - 1)) == 0 ? static_cast<int>(q) : 0;
}

#define SO_TQ_DISPATCH(TQ, CALL)           \
    switch (TQ) {                          \
    case 1: CALL(1); break;                \
    case 2: CALL(2); break;                \
    case 4: CALL(4); break;                \
    case 8: CALL(8); break;                \
    case 16: CALL(16); break;              \
    case 32: CALL(32); break;              \
    default: CALL(0); break;               \
    }

cudaError_t csr_check(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                      int full_rows, const int64_t* ls, int ls_per_coord, int64_t t, int64_t* rows_list,
                      int32_t* ent_row, int32_t* ent_gap, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_check", s);
    if (full_rows) {
        const int blocks = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>((std::max(r, nnz / 4) + kBlock - 1) / kBlock, int64_t(SO_CSR_FULL_BLOCKS_PER_SM) * num_sms())));
        launch(k_csr_check_full, dim3(blocks), dim3(kBlock), s, row_off, cols, r, c, nnz, ls_per_coord ? nullptr : ls, t,
               rows_list, d_err);
        return cudaGetLastError();
    }
    const int tq = full_row_team(c, aligned16(cols));
#define SO_CHECK(T)                                                                                              \
    launch(k_csr_check<T>,                                                                                      \
           dim3(group_blocks(r, SO_CSR_CHECK_BLOCKS_PER_SM)),                                                   \
           dim3(kBlock), s, row_off, cols, r, c, nnz, ls, ls_per_coord, t, ent_row, ent_gap, d_err)
    SO_TQ_DISPATCH(tq, SO_CHECK)
#undef SO_CHECK
    return cudaGetLastError();
}

cudaError_t csr_adam(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r, int64_t c,
                     int64_t nnz, const AdamParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_update_adam", s);
    const int tq = full_row_team(c, aligned16(vals) && aligned16(P.p) && aligned16(P.m) && aligned16(P.v) &&
                                        (!P.ls_per_coord || aligned16(P.ls)));
#define SO_ADAM(T)                                                                                               \
    launch(k_csr_update<CsrAdamOp, AdamEpi, T>, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, vals, r, c, \
           nnz, CsrAdamOp{P, c}, AdamEpi{P, c}, d_err)
    SO_TQ_DISPATCH(tq, SO_ADAM)
#undef SO_ADAM
    return cudaGetLastError();
}

cudaError_t csr_sgd(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r, int64_t c,
                    int64_t nnz, const SgdParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_update_sgd", s);
    const int tq = full_row_team(c, aligned16(vals) && aligned16(P.p) && (!P.buf || aligned16(P.buf)));
#define SO_SGD(T)                                                                                                \
    launch(k_csr_update<CsrSgdOp, SgdEpi, T>, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, vals, r, c,   \
           nnz, CsrSgdOp{P, c}, SgdEpi{P, c}, d_err)
    SO_TQ_DISPATCH(tq, SO_SGD)
#undef SO_SGD
    return cudaGetLastError();
}

// Moment state at the listed coordinates of a CSR gradient (the step's read
// set): m not finite, or v not finite or below zero, sets SPARSE_ERR_BAD_STATE.
// Runs after the structure check on the same error word and does nothing once
// that word is set, so it never follows malformed offsets or columns.
__global__ void __launch_bounds__(kBlock) k_check_state_csr(const int64_t* __restrict__ row_off,
                                                            const int32_t* __restrict__ cols, int64_t r, int64_t c,
                                                            int64_t nnz, const float* __restrict__ m,
                                                            const float* __restrict__ v, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int lane = threadIdx.x & 31;
    const int64_t groups = (r + 31) / 32;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * (kBlock / 32);
    bool bad = false;
    for (int64_t gi = static_cast<int64_t>(blockIdx.x) * (kBlock / 32) + threadIdx.x / 32; gi < groups;
         gi += gstride) {
        const int64_t r0 = gi * 32;
        const Group G = load_group(row_off, r, nnz, r0, lane);
        if (!G.ok) continue;
        for (int64_t base = G.lo; base < G.hi; base += 32) {
            const int64_t j = base + lane;
            const int l = row_lane(G, j);
            if (j < G.hi) {
                const int64_t col = cols[j];
                if (col >= 0 && col < c) {
                    const int64_t i = (r0 + l) * c + col;
                    const float mv = m[i], vv = v[i];
                    bad |= !isfinite(mv) || !isfinite(vv) || vv < 0.0f;
                }
            }
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(d_err, SPARSE_ERR_BAD_STATE);
}

cudaError_t check_state_csr(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                            const float* m, const float* v, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("check_state_csr", s);
    launch(k_check_state_csr, dim3(group_blocks(r)), dim3(kBlock), s, row_off, cols, r, c, nnz, m, v, d_err);
    return cudaGetLastError();
}

// Element-granular update from the check's per-entry rows (and gaps): one entry
// per thread, kFlatIlp entries requested at once, no walk over the rows and no
// read of last_step (the check read it; it is only rewritten here).
constexpr int kFlatIlp = 4;

struct FlatAdamOp {
    AdamParams P;
    __device__ __forceinline__ void apply(int64_t off, int32_t gap, float g, float& p, float& m, float& v) const
    {
        float b1 = P.beta1, b2 = P.beta2;
        if (P.dd) dormancy_factors(P, gap, b1, b2);
        adam_coord(P, b1, b2, g, p, m, v);
        P.p[off] = p;
        P.m[off] = m;
        P.v[off] = v;
        P.ls[off] = P.t;
    }
    __device__ __forceinline__ void load(int64_t off, float& p, float& m, float& v) const
    {
        p = P.p[off];
        m = P.m[off];
        v = P.v[off];
    }
};

struct FlatSgdOp {
    SgdParams P;
    __device__ __forceinline__ void apply(int64_t off, int32_t, float g, float& p, float& b, float&) const
    {
        sgd_coord(P, g, p, b);
        P.p[off] = p;
        if (P.buf) P.buf[off] = b;
    }
    __device__ __forceinline__ void load(int64_t off, float& p, float& b, float&) const
    {
        p = P.p[off];
        b = P.buf ? P.buf[off] : 0.0f;
    }
};

template <class Op>
__global__ void __launch_bounds__(kBlock) k_csr_flat(const int32_t* __restrict__ cols, const float* __restrict__ vals,
                                                     const int32_t* __restrict__ ent_row,
                                                     const int32_t* __restrict__ ent_gap, int64_t c, int64_t nnz,
                                                     Op op, int32_t* d_err)
{
    pdl_enter();
    if (read_error(d_err)) return;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t j0 = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; j0 < nnz; j0 += stride * kFlatIlp) {
        int64_t off[kFlatIlp];
        int32_t gap[kFlatIlp];
        float g[kFlatIlp], x0[kFlatIlp], x1[kFlatIlp], x2[kFlatIlp];
#pragma unroll
        for (int u = 0; u < kFlatIlp; ++u) {
            const int64_t j = j0 + u * stride;
            if (j < nnz) {
                off[u] = static_cast<int64_t>(__ldcs(ent_row + j)) * c + __ldcs(cols + j);
                g[u] = __ldcs(vals + j);
                gap[u] = ent_gap ? __ldcs(ent_gap + j) : 1;
            }
        }
#pragma unroll
        for (int u = 0; u < kFlatIlp; ++u)
            if (j0 + u * stride < nnz) op.load(off[u], x0[u], x1[u], x2[u]);
#pragma unroll
        for (int u = 0; u < kFlatIlp; ++u)
            if (j0 + u * stride < nnz) op.apply(off[u], gap[u], g[u], x0[u], x1[u], x2[u]);
    }
}

static int flat_grid(int64_t nnz)
{
    const int64_t want = (nnz + static_cast<int64_t>(kBlock) * kFlatIlp - 1) / (static_cast<int64_t>(kBlock) * kFlatIlp);
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 8 * num_sms())));
}

cudaError_t csr_adam_flat(const int32_t* cols, const float* vals, const int32_t* ent_row, const int32_t* ent_gap,
                          int64_t c, int64_t nnz, const AdamParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_flat_adam", s);
    launch(k_csr_flat<FlatAdamOp>, dim3(flat_grid(nnz)), dim3(kBlock), s, cols, vals, ent_row, P.dd ? ent_gap : nullptr,
           c, nnz, FlatAdamOp{P}, d_err);
    return cudaGetLastError();
}

cudaError_t csr_sgd_flat(const int32_t* cols, const float* vals, const int32_t* ent_row, int64_t c, int64_t nnz,
                         const SgdParams& P, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE("csr_flat_sgd", s);
    launch(k_csr_flat<FlatSgdOp>, dim3(flat_grid(nnz)), dim3(kBlock), s, cols, vals, ent_row, nullptr, c, nnz,
           FlatSgdOp{P}, d_err);
    return cudaGetLastError();
}

// CsrGradient::to_coo: lin[j] = row(j)*c + cols[j].
__global__ void __launch_bounds__(kBlock) k_csr_to_coo(const int64_t* __restrict__ row_off,
                                                       const int32_t* __restrict__ cols, int64_t r, int64_t c,
                                                       int64_t nnz, int64_t* __restrict__ lin, int32_t* d_err)
{
    pdl_wait();   // writes a caller output: dependents start after this grid exits
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
    pdl_wait();   // writes caller outputs: dependents start after this grid exits
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
    pdl_wait();   // writes a caller output: dependents start after this grid exits
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
