// fused.cuh -- row-fused segmented sum + optimizer update (one pass over HBM).
//
// A "team" of T lanes (T | 32) owns one table row at a time; lane tl of the team
// holds NV vectors of V floats (V = 4: 128-bit loads, used when c % 4 == 0 and
// every array is 16-byte aligned), columns col0 + (k*T + tl)*V, k < NV.  A row
// wider than T*NV*V columns is walked in chunks.
//
// Work items are "pieces": runs of at most kPieceLen sorted entries of one
// segment (one unique index).  A piece whose segment is entirely inside it is
// summed and applied directly: the team loads the row's optimizer state and the
// piece's gradient rows together, sums the gradient with error-free TwoSum
// compensation, updates and stores.  A segment that spans several pieces (a
// heavy Zipf head) is reduced by a deterministic tree: every piece writes a
// compensated partial (sum, error) to a slot, and the last of each group of
// kGroup pieces to arrive (atomic counter) combines the group's partials in
// slot order; the last group combiner of the last level applies the update.
// The order of every addition is fixed, so results are bit-reproducible, and
// no thread ever waits on another.
//
// Sum of duplicates per "DiskSparseAdam (DSA)" README, "Safe Duplicate
// Aggregation"; update rules per "Module sparse_optimizer" (optirs-gpu 0.3.2
// docs), "Lazy Adam" and "Sparse SGD".
#pragma once

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "profile.cuh"

namespace so {

// Blocks of kBlock threads per SM the fused kernel is compiled for (3: at most
// 80 registers, 24 warps per SM) and gradient rows each lane keeps in flight
// while summing a piece.  Overridable at build time for tuning sweeps.
#ifndef SO_FUSED_MIN_BLOCKS
#define SO_FUSED_MIN_BLOCKS 3
#endif
#ifndef SO_GRAD_BATCH
#define SO_GRAD_BATCH 2
#endif
constexpr int kFusedMinBlocks = SO_FUSED_MIN_BLOCKS;
constexpr int kGradBatch = SO_GRAD_BATCH;

struct PieceInfo {
    int64_t start, end;   // sorted positions [start, end)
    int64_t key;          // table row
    uint32_t u;           // segment index (row of a canonical output)
    bool multi;           // segment spans several pieces
    uint32_t perm0;       // input position of the first entry
};

// Pieces of a raw input, from the sort and run detection.
struct SortedSrc {
    const uint4* rec;
    const uint32_t* sperm;
    const uint32_t* seg_off;
    const uint32_t* counts;
    __device__ __forceinline__ int64_t count() const { return counts[kCntP]; }
    __device__ __forceinline__ PieceInfo piece(int64_t j) const
    {
        const uint4 r = rec[j];
        const uint32_t e = rec[j + 1].x;
        PieceInfo p;
        p.start = r.x;
        p.end = e;
        p.key = r.y;
        p.u = r.z & kSingleMask;
        p.multi = (r.z & kMultiFlag) != 0u;
        p.perm0 = r.w;
        return p;
    }
    __device__ __forceinline__ uint32_t perm(int64_t e) const { return sperm[e]; }
    __device__ __forceinline__ void seg_bounds(uint32_t u, int64_t& s0, int64_t& s1) const
    {
        s0 = seg_off[u];
        s1 = seg_off[u + 1];
    }
};

// Canonical row-COO: one piece per listed row, gradient row i at input row i.
struct CanonSrc {
    const int64_t* rows;
    int64_t n;
    __device__ __forceinline__ int64_t count() const { return n; }
    __device__ __forceinline__ PieceInfo piece(int64_t j) const
    {
        PieceInfo p;
        p.start = j;
        p.end = j + 1;
        p.key = rows[j];
        p.u = static_cast<uint32_t>(j);
        p.multi = false;
        p.perm0 = static_cast<uint32_t>(j);
        return p;
    }
    __device__ __forceinline__ uint32_t perm(int64_t e) const { return static_cast<uint32_t>(e); }
    __device__ __forceinline__ void seg_bounds(uint32_t, int64_t& s0, int64_t& s1) const { s0 = s1 = 0; }
};

// ------------------------------------------------------------ vector memory ops
template <int V>
__device__ __forceinline__ void ld_state(const float* p, float (&x)[V])
{
    if constexpr (V == 4) {
        const float4 a = *reinterpret_cast<const float4*>(p);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[i] = p[i];
    }
}

template <int V>
__device__ __forceinline__ void st_state(float* p, const float (&x)[V])
{
    if constexpr (V == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) p[i] = x[i];
    }
}

// gradient rows are read once: streaming (evict-first) loads
template <int V>
__device__ __forceinline__ void ld_grad(const float* p, float (&x)[V])
{
    if constexpr (V == 4) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[i] = __ldcs(p + i);
    }
}

// partials are exchanged between blocks through L2
template <int V>
__device__ __forceinline__ void ld_part(const float* p, float (&x)[V])
{
    if constexpr (V == 4) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(p));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) x[i] = __ldcg(p + i);
    }
}

template <int V>
__device__ __forceinline__ void st_part(float* p, const float (&x)[V])
{
    if constexpr (V == 4) {
        __stcg(reinterpret_cast<float4*>(p), make_float4(x[0], x[1], x[2], x[3]));
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) __stcg(p + i, x[i]);
    }
}

// ------------------------------------------------------------ the update math
// beta^gap = exp2(gap * log2(beta)), beta itself at gap 1 ("Lazy Adam",
// LazyAdamMode::DormancyDecay).
__device__ __forceinline__ void dormancy_factors(const AdamParams& P, int64_t gap, float& b1, float& b2)
{
    b1 = P.beta1;
    b2 = P.beta2;
    if (gap != 1) {
        const float gf = static_cast<float>(gap);
        b1 = exp2f(__fmul_rn(gf, P.log2b1));
        b2 = exp2f(__fmul_rn(gf, P.log2b2));
    }
}

// m = b1*m + (1-beta1)*g ; v = b2*v + (1-beta2)*g^2 ;
// p -= lr * (m / (1-beta1^t)) / (sqrt(v / (1-beta2^t)) + eps)
__device__ __forceinline__ void adam_coord(const AdamParams& P, float b1, float b2, float g, float& p,
                                           float& m, float& v)
{
    const float mi = __fmaf_rn(b1, m, __fmul_rn(P.omb1, g));
    const float vi = __fmaf_rn(b2, v, __fmul_rn(P.omb2, __fmul_rn(g, g)));
    const float m_hat = __fmul_rn(mi, P.inv_bc1);
    const float v_hat = __fmul_rn(vi, P.inv_bc2);
    const float denom = __fadd_rn(__fsqrt_rn(v_hat), P.eps);
    p = __fsub_rn(p, __fdiv_rn(__fmul_rn(P.lr, m_hat), denom));
    m = mi;
    v = vi;
}

// g' = g + wd*p ; buf = mu*buf + g' ; p -= lr*buf   (momentum 0: p -= lr*g').
// The momentum buffer is a recursion whose terms mu*buf and g often nearly
// cancel, so its new value is evaluated error-free and rounded once: mu and wd
// arrive as hi + lo float pairs (the double hyperparameters to ~2^-48), each
// product is split exactly with an FMA (TwoProduct), the three terms are added
// with TwoSum, and the accumulated low parts are added last.  The parameter
// update uses the unrounded buffer value (hi + tail).
__device__ __forceinline__ void sgd_coord(const SgdParams& P, float g, float& p, float& b)
{
    if (P.momentum != 0.0f || P.momentum_lo != 0.0f) {
        const float mh = __fmul_rn(P.momentum, b);
        const float ml = __fmaf_rn(P.momentum_lo, b, __fmaf_rn(P.momentum, b, -mh));
        const float wh = __fmul_rn(P.wd, p);
        const float wl = __fmaf_rn(P.wd_lo, p, __fmaf_rn(P.wd, p, -wh));
        float s = mh, e = ml;
        two_sum_acc(s, e, g);
        two_sum_acc(s, e, wh);
        const float tail = __fadd_rn(e, wl);
        b = __fadd_rn(s, tail);
        p = __fmaf_rn(-P.lr, tail, __fmaf_rn(-P.lr, s, p));
    } else {
        p = __fmaf_rn(-P.lr, __fmaf_rn(P.wd, p, g), p);
    }
}

// ------------------------------------------------------------ epilogues
struct AdamEpi {
    static constexpr const char* kName = "fused_rows_adam";
    AdamParams P;
    int64_t c;
    struct Row {
        int64_t key;
        float b1, b2;
    };
    template <int V>
    struct State {
        float p[V], m[V], v[V];
    };
    __device__ __forceinline__ Row begin_row(const PieceInfo& pc) const
    {
        Row r;
        r.key = pc.key;
        r.b1 = P.beta1;
        r.b2 = P.beta2;
        if (P.dd && !P.ls_per_coord) dormancy_factors(P, P.t - P.ls[pc.key], r.b1, r.b2);
        return r;
    }
    template <int V>
    __device__ __forceinline__ void load(const Row& r, int64_t col, State<V>& s) const
    {
        const int64_t off = r.key * c + col;
        ld_state<V>(P.p + off, s.p);
        ld_state<V>(P.m + off, s.m);
        ld_state<V>(P.v + off, s.v);
    }
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, State<V>& s, const float (&g)[V]) const
    {
        const int64_t off = r.key * c + col;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float b1 = r.b1, b2 = r.b2;
            if (P.dd && P.ls_per_coord) dormancy_factors(P, P.t - P.ls[off + i], b1, b2);
            adam_coord(P, b1, b2, g[i], s.p[i], s.m[i], s.v[i]);
        }
        st_state<V>(P.p + off, s.p);
        st_state<V>(P.m + off, s.m);
        st_state<V>(P.v + off, s.v);
        if (P.ls_per_coord) {
#pragma unroll
            for (int i = 0; i < V; ++i) P.ls[off + i] = P.t;
        }
    }
    // every lane of the team has read last_step before lane 0 overwrites it
    __device__ __forceinline__ void end_row(const Row& r, int tl, unsigned tmask) const
    {
        if (!P.ls_per_coord) {
            __syncwarp(tmask);
            if (tl == 0) P.ls[r.key] = P.t;
        }
    }
};

struct SgdEpi {
    static constexpr const char* kName = "fused_rows_sgd";
    SgdParams P;
    int64_t c;
    struct Row {
        int64_t key;
    };
    template <int V>
    struct State {
        float p[V], b[V];
    };
    __device__ __forceinline__ Row begin_row(const PieceInfo& pc) const { return Row{pc.key}; }
    template <int V>
    __device__ __forceinline__ void load(const Row& r, int64_t col, State<V>& s) const
    {
        const int64_t off = r.key * c + col;
        ld_state<V>(P.p + off, s.p);
        if (P.buf) ld_state<V>(P.buf + off, s.b);
    }
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, State<V>& s, const float (&g)[V]) const
    {
        const int64_t off = r.key * c + col;
#pragma unroll
        for (int i = 0; i < V; ++i) sgd_coord(P, g[i], s.p[i], s.b[i]);
        st_state<V>(P.p + off, s.p);
        if (P.buf) st_state<V>(P.buf + off, s.b);
    }
    __device__ __forceinline__ void end_row(const Row&, int, unsigned) const {}
};

// canonicalisation: write the summed row u
struct StoreEpi {
    static constexpr const char* kName = "fused_rows_sum";
    StoreParams P;
    int64_t c;
    struct Row {
        int64_t u;
    };
    template <int V>
    struct State {};
    __device__ __forceinline__ Row begin_row(const PieceInfo& pc) const { return Row{pc.u}; }
    template <int V>
    __device__ __forceinline__ void load(const Row&, int64_t, State<V>&) const {}
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, State<V>&, const float (&g)[V]) const
    {
        st_state<V>(P.out + r.u * c + col, g);
    }
    __device__ __forceinline__ void end_row(const Row&, int, unsigned) const {}
};

// ------------------------------------------------------------ the kernel
// Sum the gradient rows of entries [start, end) at this lane's columns of the
// chunk starting at col0.  The first entry initialises the sum (so a lone value
// passes through bit for bit); the compensation starts at -0.0 (s + -0.0 == s).
template <int T, int NV, int V, class Src>
__device__ __forceinline__ void sum_piece(const Src& src, const float* __restrict__ vals, int64_t c,
                                          int64_t col0, int tl, const PieceInfo& pc, float (&s)[NV][V],
                                          float (&cm)[NV][V])
{
    constexpr int B = NV >= kGradBatch ? 1 : kGradBatch / NV;   // gradient rows in flight per lane
    {
        const float* row = vals + static_cast<int64_t>(pc.perm0) * c;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
            if (col < c) ld_grad<V>(row + col, s[k]);
#pragma unroll
            for (int i = 0; i < V; ++i) cm[k][i] = -0.0f;
        }
    }
    for (int64_t e = pc.start + 1; e < pc.end; e += B) {
        uint32_t pe[B];
#pragma unroll
        for (int b = 0; b < B; ++b) pe[b] = (e + b < pc.end) ? src.perm(e + b) : 0u;
        float x[B][NV][V];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (e + b < pc.end) {
                const float* row = vals + static_cast<int64_t>(pe[b]) * c;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) ld_grad<V>(row + col, x[b][k]);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (e + b < pc.end) {
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int i = 0; i < V; ++i) two_sum_acc(s[k][i], cm[k][i], x[b][k][i]);
            }
        }
    }
}

// Slot of level-0 piece i (i-th piece, in sorted order) of the segment starting
// at sorted position s0.  Pieces after the first start at multiples of
// kPieceLen, so piece i >= 1 takes slot s0/kPieceLen + i; the first piece takes
// slot s0/kPieceLen when it starts on a multiple, else nb + s0/kPieceLen (only
// one segment can cross out of a block of kPieceLen positions).  2*nb slots.
struct SlotMap {
    int64_t b0, first;
    __device__ __forceinline__ SlotMap(int64_t s0, int64_t nb)
        : b0(s0 / kPieceLen), first((s0 % kPieceLen == 0) ? s0 / kPieceLen : nb + s0 / kPieceLen) {}
    __device__ __forceinline__ int64_t operator()(int64_t i) const { return i == 0 ? first : b0 + i; }
};

// Combining tree of a multi-piece segment, entered after this team has written
// its level-0 partial.  At each level the team bumps its group's counter; only
// the last of the group to arrive continues: it sums the group's partials in
// slot order into the slot of the group's first member (whose partial it has
// just consumed), and at the top level applies the update instead.
template <int T, int NV, int V, class Src, class Epi>
__device__ __forceinline__ void combine_tree(const Src& src, int64_t c, const Epi& epi, float* __restrict__ part,
                                             uint32_t* __restrict__ lvl_cnt, int64_t nb, const PieceInfo& pc,
                                             int tl, unsigned tmask)
{
    constexpr int CW = T * NV * V;
    const int nchunks = static_cast<int>((c + CW - 1) / CW);
    const int64_t nslots = 2 * nb;
    int64_t s0, s1;
    src.seg_bounds(pc.u, s0, s1);
    const SlotMap slot_of(s0, nb);
    int64_t Kl = 1 + (s1 - 1) / kPieceLen - slot_of.b0;   // items at this level
    int64_t kl = (pc.start == s0) ? 0 : pc.start / kPieceLen - slot_of.b0;
    int64_t stride = 1;                                   // level-0 pieces per item
    for (int lvl = 0;; ++lvl) {
        __threadfence();
        __syncwarp(tmask);
        const int64_t g = kl / kGroup;
        const int64_t members = (Kl - g * kGroup) < kGroup ? (Kl - g * kGroup) : kGroup;
        const int64_t lead_slot = slot_of(g * kGroup * stride);
        uint32_t old = 0;
        if (tl == 0) old = atomicAdd(lvl_cnt + lvl * nslots + lead_slot, 1u);
        old = __shfl_sync(tmask, old, 0, T);
        if (static_cast<int64_t>(old) != members - 1) return;   // not the last of its group
        __threadfence();
        const int64_t Knext = (Kl + kGroup - 1) / kGroup;
        const bool final = (Knext == 1);
        typename Epi::Row row{};
        if (final) row = epi.begin_row(pc);
        for (int cc = 0; cc < nchunks; ++cc) {
            const int64_t col0 = static_cast<int64_t>(cc) * CW;
            float S[NV][V], C[NV][V];
            typename Epi::template State<V> st[NV];
            if (final) {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) epi.template load<V>(row, col, st[k]);
                }
            }
            for (int64_t mi = 0; mi < members; ++mi) {
                const float* ps = part + (slot_of((g * kGroup + mi) * stride) * 2) * c;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) {
                        float xs[V], xc[V];
                        ld_part<V>(ps + col, xs);
                        ld_part<V>(ps + c + col, xc);
#pragma unroll
                        for (int i = 0; i < V; ++i) {
                            if (mi == 0) {
                                S[k][i] = xs[i];
                                C[k][i] = xc[i];
                            } else {
                                two_sum_merge(S[k][i], C[k][i], xs[i], xc[i]);
                            }
                        }
                    }
                }
            }
            float* pd = part + (lead_slot * 2) * c;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                if (col < c) {
                    if (final) {
                        float gsum[V];
#pragma unroll
                        for (int i = 0; i < V; ++i) gsum[i] = __fadd_rn(S[k][i], C[k][i]);
                        epi.template apply<V>(row, col, st[k], gsum);
                    } else {
                        st_part<V>(pd + col, S[k]);
                        st_part<V>(pd + c + col, C[k]);
                    }
                }
            }
        }
        if (final) {
            epi.end_row(row, tl, tmask);
            return;
        }
        kl = g;
        Kl = Knext;
        stride *= kGroup;
    }
}

template <int T, int NV, int V, class Src, class Epi>
__global__ void __launch_bounds__(kBlock, kFusedMinBlocks) k_fused_rows(Src src, const float* __restrict__ vals,
                                                                        int64_t c, Epi epi, float* __restrict__ part,
                                                                        uint32_t* __restrict__ lvl_cnt, int64_t nb,
                                                                        int32_t* d_err)
{
    if (read_error(d_err)) return;
    constexpr int CW = T * NV * V;
    constexpr int kTeams = kBlock / T;
    const int lane = threadIdx.x & 31;
    const int tl = lane & (T - 1);
    const unsigned tmask = (T == 32) ? kFull : (((1u << T) - 1u) << (lane & ~(T - 1)));
    const int64_t nteams = static_cast<int64_t>(gridDim.x) * kTeams;
    const int64_t P = src.count();
    const int nchunks = static_cast<int>((c + CW - 1) / CW);

    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kTeams + threadIdx.x / T; j < P; j += nteams) {
        const PieceInfo pc = src.piece(j);
        // single: the whole segment is this piece -> update directly;
        // multi: write this piece's compensated partial to its level-0 slot
        typename Epi::Row row{};
        if (!pc.multi) row = epi.begin_row(pc);
        float* ps = nullptr;
        if (pc.multi) {
            int64_t s0, s1;
            src.seg_bounds(pc.u, s0, s1);
            const SlotMap slot_of(s0, nb);
            ps = part + slot_of(pc.start == s0 ? 0 : pc.start / kPieceLen - slot_of.b0) * 2 * c;
        }
        for (int cc = 0; cc < nchunks; ++cc) {
            const int64_t col0 = static_cast<int64_t>(cc) * CW;
            typename Epi::template State<V> st[NV];
            if (!pc.multi) {
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) epi.template load<V>(row, col, st[k]);
                }
            }
            float s[NV][V], cm[NV][V];
            sum_piece<T, NV, V>(src, vals, c, col0, tl, pc, s, cm);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                if (col < c) {
                    if (!pc.multi) {
                        float g[V];
#pragma unroll
                        for (int i = 0; i < V; ++i) g[i] = __fadd_rn(s[k][i], cm[k][i]);
                        epi.template apply<V>(row, col, st[k], g);
                    } else {
                        st_part<V>(ps + col, s[k]);
                        st_part<V>(ps + c + col, cm[k]);
                    }
                }
            }
        }
        if (!pc.multi)
            epi.end_row(row, tl, tmask);
        else
            combine_tree<T, NV, V>(src, c, epi, part, lvl_cnt, nb, pc, tl, tmask);
    }
}

// ------------------------------------------------------------ launch
template <int T, int NV, int V, class Src, class Epi>
cudaError_t launch_shape(const Src& src, int64_t max_pieces, const float* vals, int64_t c, const Epi& epi,
                         float* part, uint32_t* lvl_cnt, int64_t nb, int32_t* d_err, cudaStream_t s)
{
    static int occ = 0;
    if (occ == 0) {
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_fused_rows<T, NV, V, Src, Epi>, kBlock, 0);
        if (occ <= 0) occ = 1;
    }
    constexpr int kTeams = kBlock / T;
    const int64_t want = (max_pieces + kTeams - 1) / kTeams;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)occ * num_sms())));
    SO_PROFILE(Epi::kName, s);
    k_fused_rows<T, NV, V, Src, Epi><<<blocks, kBlock, 0, s>>>(src, vals, c, epi, part, lvl_cnt, nb, d_err);
    return cudaGetLastError();
}

// Team shape: smallest power-of-two team that covers a row with one vector per
// lane; rows wider than 32 vectors give each lane up to 8 vectors per chunk.
template <class Src, class Epi>
cudaError_t launch_fused(const Src& src, int64_t max_pieces, const float* vals, int64_t c, const Epi& epi,
                         float* part, uint32_t* lvl_cnt, int64_t nb, int vec4, int32_t* d_err,
                         cudaStream_t s)
{
    if (max_pieces <= 0) return cudaSuccess;
#define SO_LAUNCH(T, NV, V) launch_shape<T, NV, V>(src, max_pieces, vals, c, epi, part, lvl_cnt, nb, d_err, s)
    if (vec4) {
        const int64_t nv = c / 4;
        if (nv <= 1) return SO_LAUNCH(1, 1, 4);
        if (nv <= 2) return SO_LAUNCH(2, 1, 4);
        if (nv <= 4) return SO_LAUNCH(4, 1, 4);
        if (nv <= 8) return SO_LAUNCH(8, 1, 4);
        if (nv <= 16) return SO_LAUNCH(16, 1, 4);
        if (nv <= 32) return SO_LAUNCH(32, 1, 4);
        if (nv <= 64) return SO_LAUNCH(32, 2, 4);
        if (nv <= 128) return SO_LAUNCH(32, 4, 4);
        return SO_LAUNCH(32, 8, 4);
    }
    if (c <= 1) return SO_LAUNCH(1, 1, 1);
    if (c <= 2) return SO_LAUNCH(2, 1, 1);
    if (c <= 4) return SO_LAUNCH(4, 1, 1);
    if (c <= 8) return SO_LAUNCH(8, 1, 1);
    if (c <= 16) return SO_LAUNCH(16, 1, 1);
    if (c <= 32) return SO_LAUNCH(32, 1, 1);
    return SO_LAUNCH(32, 4, 1);
#undef SO_LAUNCH
}

inline SortedSrc sorted_src(const SortWs& ws)
{
    return SortedSrc{ws.rec, ws.vals[ws.final_buf], ws.seg_off, ws.counts};
}

}  // namespace so
