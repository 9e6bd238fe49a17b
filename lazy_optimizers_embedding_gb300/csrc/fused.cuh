// fused.cuh -- row-fused segmented sum + optimizer update (one pass over HBM).
//
// A "team" of T lanes (T | 32) owns one table row at a time; lane tl of the team
// holds NV vectors of V floats (V = 4: 128-bit loads, used when c % 4 == 0 and
// every array is 16-byte aligned), columns col0 + (k*T + tl)*V, k < NV.  A row
// wider than T*NV*V columns is walked in chunks.
//
// Work items are "pieces": runs of fewer than 2*kPieceLen sorted entries of one
// segment (one unique index); a segment of at most kPieceLen entries is always
// a single piece.  A piece whose segment is entirely inside it is summed and
// applied directly: the team loads the row's optimizer state and the piece's
// gradient rows together, sums the gradient with error-free TwoSum
// compensation, updates and stores.  A segment that spans several pieces (a
// heavy Zipf head) is reduced in a second launch: the row kernel writes every
// piece's compensated partial (sum, error) to a slot, then the combine kernel
// merges groups of kGroup consecutive pieces (one team each) and the last group
// of each segment to finish merges the groups and applies the update.  The
// order of every addition is fixed, so results are bit-reproducible, and no
// thread ever waits on another.
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

// Blocks of kRowBlock threads per SM the row kernel is compiled for (3 of 256:
// at most 80 registers, 24 warps per SM), short pieces per work ticket
// (kTicket), gradient rows a lane requests at once (kRowIlp, kLongIlp), rows of
// a long piece staged in shared memory per round (kLongStage), threads of a
// combine block and the partial pairs a thread of it requests at once when they
// are not staged (kCombineIlp).  Overridable at build time for tuning sweeps.
#ifndef SO_FUSED_MIN_BLOCKS
#define SO_FUSED_MIN_BLOCKS 3
#endif
#ifndef SO_TICKET
#define SO_TICKET 4
#endif
#ifndef SO_ROW_ILP
#define SO_ROW_ILP 3
#endif
#ifndef SO_LONG_ILP
#define SO_LONG_ILP 4
#endif
#ifndef SO_COMBINE_ILP
#define SO_COMBINE_ILP 8
#endif
#ifndef SO_ROW_BLOCK
#define SO_ROW_BLOCK 256
#endif
constexpr int kRowBlock = SO_ROW_BLOCK;   // threads of a row-kernel block
#ifndef SO_LONG_STAGE
#define SO_LONG_STAGE 8
#endif
// Gradient rows of a long piece a team stages in shared memory per round (0:
// the rows are requested into registers, kLongIlp at a time).
constexpr int kLongStage = SO_LONG_STAGE;
constexpr int kFusedMinBlocks = SO_FUSED_MIN_BLOCKS;
constexpr int kTicket = SO_TICKET;
constexpr int kRowIlp = SO_ROW_ILP;
constexpr int kLongIlp = SO_LONG_ILP;   // gradient rows requested at once in a long piece (unstaged shapes)
constexpr int kCombineBlock = 128;
// Combine groups staged through shared memory (1) or merged from registers only (0).
#ifndef SO_COMBINE_STAGED
#define SO_COMBINE_STAGED 1
#endif
constexpr int kCombineIlp = SO_COMBINE_ILP;

struct PieceInfo {
    uint32_t start, end;  // sorted positions [start, end)
    uint32_t key;         // table row (< 2^32: raw keys and canonical rows both are)
    uint32_t uf;          // segment index (row of a canonical output) | flags
    uint32_t perm0;       // input position of the first entry
    // kMultiFlag: segment spans several pieces; kLongFlag: one long piece
    __device__ __forceinline__ uint32_t u() const { return uf & kSingleMask; }
    __device__ __forceinline__ uint32_t flags() const { return uf & (kMultiFlag | kLongFlag); }
    __device__ __forceinline__ bool multi() const { return (uf & kMultiFlag) != 0u; }
    __device__ __forceinline__ bool is_short() const { return (uf & (kMultiFlag | kLongFlag)) == 0u; }
};

// Pieces of a raw input, from the sort and run detection.
struct SortedSrc {
    const uint4* rec;
    const uint32_t* sperm;
    const uint32_t* seg_off;
    const uint32_t* mlist;
    const uint32_t* slist;
    const uint32_t* glist;
    const uint32_t* counts;
    uint32_t* scnt;   // groups of a split segment merged so far (by its first piece's slot)
    __device__ __forceinline__ int64_t count() const { return counts[kCntP]; }
    __device__ __forceinline__ int64_t count_multi() const { return counts[kCntM]; }
    __device__ __forceinline__ int64_t multi_index(int64_t t) const { return mlist[t]; }
    __device__ __forceinline__ int64_t count_split() const { return counts[kCntS]; }
    __device__ __forceinline__ int64_t split_index(int64_t t) const { return slist[t]; }
    __device__ __forceinline__ int64_t count_groups() const { return counts[kCntG]; }
    __device__ __forceinline__ int64_t group_index(int64_t t) const { return glist[t]; }
    __device__ __forceinline__ uint32_t* segment_counter(int64_t slot) const { return scnt + slot; }
    static constexpr bool kTickets = true;
    __device__ __forceinline__ uint32_t* ticket(int which) const { return const_cast<uint32_t*>(counts) + which; }
    __device__ __forceinline__ PieceInfo piece(int64_t j) const
    {
        const uint4 r = rec[j];
        const uint32_t e = rec[j + 1].x;
        PieceInfo p;
        p.start = r.x;
        p.end = e;
        p.key = r.y;
        p.uf = r.z;
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
    __device__ __forceinline__ int64_t count_multi() const { return 0; }
    __device__ __forceinline__ int64_t multi_index(int64_t) const { return 0; }
    __device__ __forceinline__ int64_t count_split() const { return 0; }
    __device__ __forceinline__ int64_t split_index(int64_t) const { return 0; }
    __device__ __forceinline__ int64_t count_groups() const { return 0; }
    __device__ __forceinline__ int64_t group_index(int64_t) const { return 0; }
    __device__ __forceinline__ uint32_t* segment_counter(int64_t) const { return nullptr; }
    static constexpr bool kTickets = false;
    __device__ __forceinline__ uint32_t* ticket(int) const { return nullptr; }
    __device__ __forceinline__ PieceInfo piece(int64_t j) const
    {
        PieceInfo p;
        p.start = static_cast<uint32_t>(j);
        p.end = static_cast<uint32_t>(j + 1);
        p.key = static_cast<uint32_t>(rows[j]);
        p.uf = static_cast<uint32_t>(j) & kSingleMask;
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

// partials are exchanged between kernels through L2
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

// Partials are written long before the combine kernels read them, with the
// whole step's gradient and state streaming through L2 in between: they are
// stored with an L2 evict-last policy so that the combine reads hit L2.
__device__ __forceinline__ uint64_t l2_keep_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <int V>
__device__ __forceinline__ void st_part(float* p, const float (&x)[V])
{
    const uint64_t pol = l2_keep_policy();
    if constexpr (V == 4) {
        asm volatile("st.global.cg.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(x[0]),
                     "f"(x[1]), "f"(x[2]), "f"(x[3]), "l"(pol)
                     : "memory");
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i)
            asm volatile("st.global.cg.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p + i), "f"(x[i]), "l"(pol) : "memory");
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
// With weight decay ("DiskSparseAdam (DSA)" README, "Explicit Weight Decay
// Semantics"): L2 adds wd*p to g first; decoupled adds wd*p to the descent
// direction, p -= lr * (m_hat / (sqrt(v_hat) + eps) + wd*p) (AdamW).
__device__ __forceinline__ void adam_coord(const AdamParams& P, float b1, float b2, float g, float& p,
                                           float& m, float& v)
{
    if (P.wd != 0.0f) {
        const float p0 = p;
        // L2: g + wd*p with wd as a hi + lo pair, so that a gradient nearly cancelled by
        // the decay term keeps its relative accuracy (the product is exact inside the FMA)
        if (!P.wd_decoupled) g = __fmaf_rn(P.wd_lo, p0, __fmaf_rn(P.wd, p0, g));
        const float mi = __fmaf_rn(b1, m, __fmul_rn(P.omb1, g));
        const float vi = __fmaf_rn(b2, v, __fmul_rn(P.omb2, __fmul_rn(g, g)));
        const float m_hat = __fmul_rn(mi, P.inv_bc1);
        const float v_hat = __fmul_rn(vi, P.inv_bc2);
        const float denom = __fadd_rn(__fsqrt_rn(v_hat), P.eps);
        float dir = __fdiv_rn(m_hat, denom);
        if (P.wd_decoupled) dir = __fmaf_rn(P.wd, p0, dir);
        p = __fsub_rn(p0, __fmul_rn(P.lr, dir));
        m = mi;
        v = vi;
        return;
    }
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
// An epilogue owns the optimizer state of a row: kArrays fp32 arrays of r*c
// values (arrays() of them live), read at the row's columns, updated from the
// summed gradient and written back; optionally one int64 per row (last_step)
// read before the update (stage_last) and rewritten after it (end_row).
struct AdamEpi {
    static constexpr const char* kName = "fused_rows_adam";
    static constexpr const char* kCombineName = "combine_split_adam";
    static constexpr int kArrays = 3;   // p, m, v
    static constexpr bool kEarlyRelease = true;   // writes optimizer state only
    AdamParams P;
    int64_t c;
    struct Row {
        int64_t key;
        int64_t last;   // last_step of the row (per-row layout, DormancyDecay)
    };
    __device__ __forceinline__ const int64_t* stage_last(const PieceInfo& pc) const
    {
        return (P.dd && !P.ls_per_coord) ? P.ls + pc.key : nullptr;
    }
    __device__ __forceinline__ Row make_row(const PieceInfo& pc, int64_t last) const { return Row{pc.key, last}; }
    __device__ __forceinline__ int arrays() const { return 3; }
    __device__ __forceinline__ float* array(int a) const { return a == 0 ? P.p : (a == 1 ? P.m : P.v); }
    __device__ __forceinline__ int64_t base(const PieceInfo& pc) const { return pc.key * c; }
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, float (&x)[kArrays][V], const float (&g)[V]) const
    {
        const int64_t off = r.key * c + col;
        float rb1 = P.beta1, rb2 = P.beta2;
        if (P.dd && !P.ls_per_coord) dormancy_factors(P, P.t - r.last, rb1, rb2);
#pragma unroll
        for (int i = 0; i < V; ++i) {
            float b1 = rb1, b2 = rb2;
            if (P.dd && P.ls_per_coord) dormancy_factors(P, P.t - P.ls[off + i], b1, b2);
            adam_coord(P, b1, b2, g[i], x[0][i], x[1][i], x[2][i]);
        }
        st_state<V>(P.p + off, x[0]);
        st_state<V>(P.m + off, x[1]);
        st_state<V>(P.v + off, x[2]);
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
    static constexpr const char* kCombineName = "combine_split_sgd";
    static constexpr int kArrays = 2;   // p, momentum buffer (absent without momentum)
    static constexpr bool kEarlyRelease = true;   // writes optimizer state only
    SgdParams P;
    int64_t c;
    struct Row {
        int64_t key;
    };
    __device__ __forceinline__ const int64_t* stage_last(const PieceInfo&) const { return nullptr; }
    __device__ __forceinline__ Row make_row(const PieceInfo& pc, int64_t) const { return Row{pc.key}; }
    __device__ __forceinline__ int arrays() const { return P.buf ? 2 : 1; }
    __device__ __forceinline__ float* array(int a) const { return a == 0 ? P.p : P.buf; }
    __device__ __forceinline__ int64_t base(const PieceInfo& pc) const { return pc.key * c; }
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, float (&x)[kArrays][V], const float (&g)[V]) const
    {
        const int64_t off = r.key * c + col;
#pragma unroll
        for (int i = 0; i < V; ++i) sgd_coord(P, g[i], x[0][i], x[1][i]);
        st_state<V>(P.p + off, x[0]);
        if (P.buf) st_state<V>(P.buf + off, x[1]);
    }
    __device__ __forceinline__ void end_row(const Row&, int, unsigned) const {}
};

// canonicalisation: write the summed row u
struct StoreEpi {
    static constexpr const char* kName = "fused_rows_sum";
    static constexpr const char* kCombineName = "combine_split_sum";
    static constexpr int kArrays = 1;   // no state; one dummy array keeps the types simple
    static constexpr bool kEarlyRelease = false;  // writes a caller output (the summed rows)
    StoreParams P;
    int64_t c;
    struct Row {
        int64_t u;
    };
    __device__ __forceinline__ const int64_t* stage_last(const PieceInfo&) const { return nullptr; }
    __device__ __forceinline__ Row make_row(const PieceInfo& pc, int64_t) const { return Row{pc.u()}; }
    __device__ __forceinline__ int arrays() const { return 0; }
    __device__ __forceinline__ float* array(int) const { return nullptr; }
    __device__ __forceinline__ int64_t base(const PieceInfo&) const { return 0; }
    template <int V>
    __device__ __forceinline__ void apply(const Row& r, int64_t col, float (&)[kArrays][V], const float (&g)[V]) const
    {
        st_state<V>(P.out + r.u * c + col, g);
    }
    __device__ __forceinline__ void end_row(const Row&, int, unsigned) const {}
};

// ------------------------------------------------------------ the kernels
// First gradient row of a piece at this lane's columns of the chunk at col0.
// It initialises the sum: a lone value passes through bit for bit.
template <int T, int NV, int V>
__device__ __forceinline__ void first_row(const float* __restrict__ vals, int64_t c, int64_t col0, int tl,
                                          uint32_t perm0, float (&s)[NV][V])
{
    const float* row = vals + static_cast<int64_t>(perm0) * c;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
        if (col < c) ld_grad<V>(row + col, s[k]);
    }
}

// The TwoSum compensation of a sum starts at -0.0 (s + -0.0 == s).
template <int NV, int V>
__device__ __forceinline__ void zero_comp(float (&cm)[NV][V])
{
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int i = 0; i < V; ++i) cm[k][i] = -0.0f;
}

// Input positions of the entries after the first of a piece (fewer than
// 2*kPieceLen of them), spread over the team and loaded in one round trip:
// lane tl holds entries start+1+tl, start+1+tl+T, ...  Teams of fewer than 8
// lanes read each position when they use it.
template <int T>
struct PiecePerms {
    static constexpr int kPerLane = T >= 8 ? (2 * kPieceLen - 2 + T - 1) / T : 1;
    uint32_t pm[kPerLane];
    template <class Src>
    __device__ __forceinline__ void load(const Src& src, const PieceInfo& pc, int tl)
    {
        if constexpr (T >= 8) {
#pragma unroll
            for (int k = 0; k < kPerLane; ++k) {
                const int64_t e = pc.start + 1 + tl + k * T;
                pm[k] = (e < pc.end) ? src.perm(e) : 0u;
            }
        }
    }
    // every lane of the team calls with the same e
    template <class Src>
    __device__ __forceinline__ uint32_t get(const Src& src, const PieceInfo& pc, int64_t e, unsigned tmask) const
    {
        if constexpr (T >= 8) {
            const int i = static_cast<int>(e - pc.start - 1);
            uint32_t v = pm[0];
#pragma unroll
            for (int k = 1; k < kPerLane; ++k)
                if (i / T == k) v = pm[k];
            return __shfl_sync(tmask, v, i % T, T);
        } else {
            return src.perm(e);
        }
    }
};

// Gradient rows start+1 .. end-1 of a piece, ILP rows requested at once, added
// in entry order with TwoSum compensation.
template <int T, int NV, int V, int ILP, class Src>
__device__ __forceinline__ void sum_rest(const Src& src, const PiecePerms<T>& pp, const float* __restrict__ vals,
                                         int64_t c, int64_t col0, int tl, unsigned tmask, const PieceInfo& pc,
                                         float (&s)[NV][V], float (&cm)[NV][V])
{
    constexpr int R = NV >= ILP ? 1 : ILP / NV;
    for (int64_t e0 = pc.start + 1; e0 < pc.end; e0 += R) {
        float x[R][NV][V];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t e = e0 + r;
            if (e < pc.end) {
                const float* row = vals + static_cast<int64_t>(pp.get(src, pc, e, tmask)) * c;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                    if (col < c) ld_grad<V>(row + col, x[r][k]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (e0 + r < pc.end) {
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int i = 0; i < V; ++i) two_sum_acc(s[k][i], cm[k][i], x[r][k][i]);
            }
        }
    }
}

// ------------------------------------------------------------ staged long pieces
// With kLongStage > 0 a long piece's gradient rows travel through the team's
// shared buffer instead of registers: every lane copies its 16 bytes of each of
// up to kLongStage rows with cp.async, waits for its own copies and adds its
// slice of the rows in entry order with TwoSum compensation, the same
// operations in the same order as sum_rest.  A lane reads back only what it
// copied itself, so no barrier is needed.  For rows of whole 16-byte vectors in
// one chunk (the float4 instantiations) and teams of 8 lanes or more.
template <int T, int NV, int V, class Src>
__host__ __device__ constexpr bool long_staged()
{
    return kLongStage > 0 && Src::kTickets && NV == 1 && V == 4 && T >= 8;
}
// dynamic shared memory of a row-kernel block: every team kLongStage rows of at most 4T floats
__host__ __device__ constexpr size_t long_stage_bytes() { return static_cast<size_t>(kRowBlock) * kLongStage * 16; }

template <int T>
__device__ __forceinline__ void staged_rest(const PiecePerms<T>& pp, const PieceInfo& pc, const float* __restrict__ vals,
                                            int64_t c, int tl, unsigned tmask, uint32_t buf_s, float (&s)[4],
                                            float (&cm)[4])
{
    const int rest = static_cast<int>(pc.end - pc.start) - 1;
    const uint32_t row_bytes = static_cast<uint32_t>(c) * 4u;
    const bool mine = tl * 4 < c;
    const uint32_t lane_s = buf_s + static_cast<uint32_t>(tl) * 16u;
    const float* lane_v = vals + tl * 4;
    for (int k0 = 0; k0 < rest; k0 += kLongStage) {
        const int cnt = (rest - k0) < kLongStage ? (rest - k0) : kLongStage;
#pragma unroll
        for (int q = 0; q < PiecePerms<T>::kPerLane; ++q) {
            // rows k0 .. k0+cnt-1 whose input positions sit in slot q of lanes 0..T-1
            const int lo = q * T > k0 ? q * T : k0;
            const int hi = (q + 1) * T < k0 + cnt ? (q + 1) * T : k0 + cnt;
            for (int i = lo; i < hi; ++i) {
                const uint32_t pr = __shfl_sync(tmask, pp.pm[q], i - q * T, T);
                if (mine)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                                     lane_s + static_cast<uint32_t>(i - k0) * row_bytes),
                                 "l"(lane_v + static_cast<int64_t>(pr) * c)
                                 : "memory");
            }
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        if (mine) {
            for (int r = 0; r < cnt; ++r) {
                float4 x;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                             : "r"(lane_s + static_cast<uint32_t>(r) * row_bytes)
                             : "memory");
                two_sum_acc(s[0], cm[0], x.x);
                two_sum_acc(s[1], cm[1], x.y);
                two_sum_acc(s[2], cm[2], x.z);
                two_sum_acc(s[3], cm[3], x.w);
            }
        }
    }
}

// Pieces of a split segment [s0, s1) and their partial-sum slots.  The first
// piece starts at s0; piece i >= 1 starts at q1 + (i-1)*kPieceLen, where q1 is
// the smallest multiple of kPieceLen >= s0 + kPieceLen (see run detection).  A
// piece starting at a multiple of kPieceLen takes slot start/kPieceLen; a first
// piece starting elsewhere takes nb + start/kPieceLen (a split segment is
// longer than kPieceLen, so no two of them start in the same block of kPieceLen
// positions).  2*nb slots in all; a slot depends on the piece's start alone.
__device__ __forceinline__ int64_t part_slot(int64_t start, int64_t nb)
{
    return (start % kPieceLen == 0) ? start / kPieceLen : nb + start / kPieceLen;
}
// Combine groups: piece i sits at the "aligned start" q1 + (i-1)*kPieceLen (its
// true start for i >= 1, a multiple of kPieceLen), and a group is the pieces
// whose aligned starts share a block of kGroup*kPieceLen positions (at most
// kGroup pieces).  Its head, the piece run detection lists, is the segment's
// first piece or the piece starting at the block boundary.
struct SplitSegment {
    int64_t s0, s1, q1;
    __device__ __forceinline__ SplitSegment(int64_t a, int64_t b)
        : s0(a), s1(b), q1((a + 2 * kPieceLen - 1) / kPieceLen * kPieceLen) {}
    __device__ __forceinline__ int64_t pieces() const { return (s1 - 1 >= q1) ? 2 + (s1 - 1 - q1) / kPieceLen : 1; }
    __device__ __forceinline__ int64_t start(int64_t i) const { return i == 0 ? s0 : q1 + (i - 1) * kPieceLen; }
    __device__ __forceinline__ int64_t index(int64_t st) const { return st == s0 ? 0 : (st - q1) / kPieceLen + 1; }
    __device__ __forceinline__ int64_t group(int64_t i) const { return (q1 + (i - 1) * kPieceLen) / kGroupSpan; }
    // index of the first piece of group g (the segment's first group: piece 0)
    __device__ __forceinline__ int64_t group_head(int64_t g) const
    {
        return g == group(0) ? 0 : (g * kGroupSpan - q1) / kPieceLen + 1;
    }
    static constexpr int64_t kGroupSpan = static_cast<int64_t>(kGroup) * kPieceLen;
};

// Loads the optimizer state of one row chunk (the live arrays of the epilogue).
template <int T, int NV, int V, class Epi>
__device__ __forceinline__ void load_state(const Epi& epi, const PieceInfo& pc, int64_t c, int64_t col0, int tl,
                                           float (&x)[NV][Epi::kArrays][V])
{
    const int na = epi.arrays();
    const int64_t rb = epi.base(pc);
#pragma unroll
    for (int a = 0; a < Epi::kArrays; ++a) {
        if (a < na) {
            const float* arr = epi.array(a) + rb;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
                if (col < c) ld_state<V>(arr + col, x[k][a]);
            }
        }
    }
}

// Adds the rest of a piece's gradient rows (if any) to the first one, applies
// the update to the row chunk at col0 and stores it.
template <int T, int NV, int V, int ILP, class Src, class Epi>
__device__ __forceinline__ void finish_chunk(const Src& src, const PiecePerms<T>& pp, const float* __restrict__ vals,
                                             int64_t c, const Epi& epi, const PieceInfo& pc,
                                             const typename Epi::Row& row, int64_t col0, int tl, unsigned tmask,
                                             float (&x)[NV][Epi::kArrays][V], float (&s)[NV][V])
{
    if (pc.end - pc.start > 1) {
        float cm[NV][V];
        zero_comp<NV, V>(cm);
        sum_rest<T, NV, V, ILP>(src, pp, vals, c, col0, tl, tmask, pc, s, cm);
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int i = 0; i < V; ++i) s[k][i] = __fadd_rn(s[k][i], cm[k][i]);
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
        if (col < c) epi.template apply<V>(row, col, x[k], s[k]);
    }
}

// One piece holding its whole segment, row chunk by row chunk: the row's state,
// last_step and first gradient row are requested together, the other gradient
// rows ILP at a time.
template <int T, int NV, int V, int ILP, class Src, class Epi>
__device__ __forceinline__ void apply_single(const Src& src, const float* __restrict__ vals, int64_t c,
                                             const Epi& epi, const PieceInfo& pc, int tl, unsigned tmask)
{
    constexpr int CW = T * NV * V;
    constexpr int A = Epi::kArrays;
    const int nchunks = static_cast<int>((c + CW - 1) / CW);
    const int64_t* lp = epi.stage_last(pc);
    int64_t last = 0;
    PiecePerms<T> pp;
    if (pc.end - pc.start > 1) pp.load(src, pc, tl);
    for (int cc = 0; cc < nchunks; ++cc) {
        const int64_t col0 = static_cast<int64_t>(cc) * CW;
        float x[NV][A][V];
        load_state<T, NV, V>(epi, pc, c, col0, tl, x);
        if (cc == 0 && lp) last = *lp;
        float s[NV][V];
        first_row<T, NV, V>(vals, c, col0, tl, pc.perm0, s);
        finish_chunk<T, NV, V, ILP>(src, pp, vals, c, epi, pc, epi.make_row(pc, last), col0, tl, tmask, x, s);
    }
    epi.end_row(epi.make_row(pc, last), tl, tmask);
}

// Lane `from` of the team's piece, for every lane of the team.
template <int T>
__device__ __forceinline__ PieceInfo shfl_piece(const PieceInfo& p, int from, unsigned tmask)
{
    PieceInfo q;
    q.start = __shfl_sync(tmask, p.start, from, T);
    q.end = __shfl_sync(tmask, p.end, from, T);
    q.key = __shfl_sync(tmask, p.key, from, T);
    q.uf = __shfl_sync(tmask, p.uf, from, T);
    q.perm0 = __shfl_sync(tmask, p.perm0, from, T);
    return q;
}

// A piece of a split segment: its compensated partial sum (sum, error) goes to
// the piece's slot, to be combined by k_combine_split.
template <int T, int NV, int V, class Src>
__device__ __forceinline__ void store_partial(const Src& src, const float* __restrict__ vals, int64_t c,
                                              float* __restrict__ part, int64_t nb, const PieceInfo& pc, int tl,
                                              unsigned tmask)
{
    constexpr int CW = T * NV * V;
    const int nchunks = static_cast<int>((c + CW - 1) / CW);
    float* ps = part + part_slot(pc.start, nb) * 2 * c;
    PiecePerms<T> pp;
    pp.load(src, pc, tl);
    for (int cc = 0; cc < nchunks; ++cc) {
        const int64_t col0 = static_cast<int64_t>(cc) * CW;
        float s[NV][V], cm[NV][V];
        first_row<T, NV, V>(vals, c, col0, tl, pc.perm0, s);
        zero_comp<NV, V>(cm);
        sum_rest<T, NV, V, kLongIlp>(src, pp, vals, c, col0, tl, tmask, pc, s, cm);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int64_t col = col0 + static_cast<int64_t>(k * T + tl) * V;
            if (col < c) {
                st_part<V>(ps + col, s[k]);
                st_part<V>(ps + c + col, cm[k]);
            }
        }
    }
}

// store_partial and apply_single for a long piece through the team's stage.
template <int T, class Src>
__device__ __forceinline__ void store_partial_staged(const Src& src, const float* __restrict__ vals, int64_t c,
                                                     float* __restrict__ part, int64_t nb, const PieceInfo& pc,
                                                     int tl, unsigned tmask, uint32_t buf_s)
{
    float* ps = part + part_slot(pc.start, nb) * 2 * c;
    PiecePerms<T> pp;
    pp.load(src, pc, tl);
    float s[1][4], cm[1][4];
    first_row<T, 1, 4>(vals, c, 0, tl, pc.perm0, s);
    zero_comp<1, 4>(cm);
    staged_rest<T>(pp, pc, vals, c, tl, tmask, buf_s, s[0], cm[0]);
    const int64_t col = static_cast<int64_t>(tl) * 4;
    if (col < c) {
        st_part<4>(ps + col, s[0]);
        st_part<4>(ps + c + col, cm[0]);
    }
}

template <int T, class Src, class Epi>
__device__ __forceinline__ void apply_single_staged(const Src& src, const float* __restrict__ vals, int64_t c,
                                                    const Epi& epi, const PieceInfo& pc, int tl, unsigned tmask,
                                                    uint32_t buf_s)
{
    const int64_t* lp = epi.stage_last(pc);
    PiecePerms<T> pp;
    if (pc.end - pc.start > 1) pp.load(src, pc, tl);
    float x[1][Epi::kArrays][4];
    load_state<T, 1, 4>(epi, pc, c, 0, tl, x);
    const int64_t last = lp ? *lp : 0;
    float s[1][4];
    first_row<T, 1, 4>(vals, c, 0, tl, pc.perm0, s);
    if (pc.end - pc.start > 1) {
        float cm[1][4];
        zero_comp<1, 4>(cm);
        staged_rest<T>(pp, pc, vals, c, tl, tmask, buf_s, s[0], cm[0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) s[0][i] = __fadd_rn(s[0][i], cm[0][i]);
    }
    const typename Epi::Row row = epi.make_row(pc, last);
    const int64_t col = static_cast<int64_t>(tl) * 4;
    if (col < c) epi.template apply<4>(row, col, x[0], s[0]);
    epi.end_row(row, tl, tmask);
}

// Every piece of the input.  On a raw input the pieces range from one to
// 2*kPieceLen-1 gradient rows.  Long pieces come first (the list run detection
// built: pieces of split segments, whose partials the combine kernel waits
// for, and whole segments of more than kShortLen entries), split statically
// over the teams, their gradient rows staged through shared memory
// (kLongStage rows a round, where the shape allows), so that the registers go
// to the short pieces' loads; then short pieces are handed out by atomic tickets, kTicket
// per ticket (their records one per lane), so that teams with less long work
// take more of them.  A team requests its next piece's record, or its next
// ticket and that ticket's records, while it works on the current ones.  A
// canonical input (one row per piece) is split statically, each team fetching
// the record of its next piece during the current one.
template <int T, int NV, int V, class Src, class Epi>
__global__ void __launch_bounds__(kRowBlock, kFusedMinBlocks) k_fused_rows(Src src, const float* __restrict__ vals,
                                                                        int64_t c, Epi epi, float* __restrict__ part,
                                                                        int64_t nb, int32_t* d_err)
{
    pdl_wait();
    if constexpr (Epi::kEarlyRelease) pdl_release();
    if (read_error(d_err)) return;
    constexpr int kTeams = kRowBlock / T;
    const int lane = threadIdx.x & 31;
    const int tl = lane & (T - 1);
    const unsigned tmask = (T == 32) ? kFull : (((1u << T) - 1u) << (lane & ~(T - 1)));
    const int64_t P = src.count();
    if constexpr (Src::kTickets) {
        const auto take = [&](int which) {
            uint32_t t = 0;
            if (tl == 0) t = atomicAdd(src.ticket(which), 1u);
            return t;
        };
        {   // long pieces
            const int64_t M = src.count_multi();
            const auto record = [&](uint32_t t, PieceInfo& r) {
                if (tl == 0 && t < M) r = src.piece(src.multi_index(t));
            };
            // team g takes long pieces g, g + teams, ...: there are about two per
            // team, and a static split spares every team the ticket round trip
            // on one counter that all of them hit at the kernel's start
            const uint32_t nteams = gridDim.x * kTeams;
            uint32_t ta = blockIdx.x * kTeams + threadIdx.x / T;
            uint32_t tb = ta + nteams;
            PieceInfo ra{}, rb{};
            record(ta, ra);
            [[maybe_unused]] uint32_t buf_s = 0;
            if constexpr (long_staged<T, NV, V, Src>()) {
                extern __shared__ float4 so_long_stage[];
                buf_s = static_cast<uint32_t>(__cvta_generic_to_shared(so_long_stage)) +
                        static_cast<uint32_t>((threadIdx.x / T) * kLongStage) * static_cast<uint32_t>(c) * 4u;
            }
            while (ta < M) {
                record(tb, rb);
                const PieceInfo pc = shfl_piece<T>(ra, 0, tmask);
                if constexpr (long_staged<T, NV, V, Src>()) {
                    if (pc.multi())
                        store_partial_staged<T>(src, vals, c, part, nb, pc, tl, tmask, buf_s);
                    else
                        apply_single_staged<T>(src, vals, c, epi, pc, tl, tmask, buf_s);
                } else if (pc.multi()) {
                    store_partial<T, NV, V>(src, vals, c, part, nb, pc, tl, tmask);
                } else {
                    apply_single<T, NV, V, kLongIlp>(src, vals, c, epi, pc, tl, tmask);
                }
                ta = tb;
                ra = rb;
                tb += nteams;
            }
        }
        {   // short pieces
            constexpr int K = kTicket < T ? kTicket : T;
            const int64_t nt = (P + K - 1) / K;
            const auto records = [&](uint32_t t, PieceInfo& r) {
                const int64_t j = static_cast<int64_t>(t) * K + tl;
                if (tl < K && j < P) r = src.piece(j);
            };
            uint32_t ta = __shfl_sync(tmask, take(kTicketS), 0, T);
            uint32_t tb = take(kTicketS);
            PieceInfo ra{}, rb{};
            records(ta, ra);
            tb = __shfl_sync(tmask, tb, 0, T);
            while (ta < nt) {
                records(tb, rb);
                const uint32_t tc = (tb < nt) ? take(kTicketS) : tb;
                const int64_t j0 = static_cast<int64_t>(ta) * K;
                const int nd = (P - j0) < K ? static_cast<int>(P - j0) : K;
                for (int d = 0; d < nd; ++d) {
                    const PieceInfo pc = shfl_piece<T>(ra, d, tmask);
                    if (pc.is_short()) apply_single<T, NV, V, kRowIlp>(src, vals, c, epi, pc, tl, tmask);
                }
                ta = tb;
                ra = rb;
                tb = __shfl_sync(tmask, tc, 0, T);
            }
        }
    } else {
        const int64_t team_g = static_cast<int64_t>(blockIdx.x) * kTeams + threadIdx.x / T;
        const int64_t nteams = static_cast<int64_t>(gridDim.x) * kTeams;
        PieceInfo mine{};
        if (team_g < P && tl == 0) mine = src.piece(team_g);
        for (int64_t j = team_g; j < P; j += nteams) {
            const PieceInfo pc = shfl_piece<T>(mine, 0, tmask);
            if (j + nteams < P && tl == 0) mine = src.piece(j + nteams);
            apply_single<T, NV, V, kRowIlp>(src, vals, c, epi, pc, tl, tmask);
        }
    }
}

// Partial slots of a run of pairs: pair 0 in slot `first`, pair k >= 1 in slot
// base + k*step (the slots of a split segment's pieces after the first are
// consecutive, those of its group heads kGroup apart).
struct SlotRun {
    int64_t first, base, step, cnt;
    __device__ __forceinline__ int64_t slot(int64_t k) const { return k == 0 ? first : base + k * step; }
};

// Columns a combine block merges per round through its shared stage, and the
// pairs it stages per round: by default one group's worth, so that merging a
// group costs one round trip (a 16-pair stage, 16 KB at 128 columns, measured
// faster than 32-pair ones, whose 32 KB make the SMs change their shared-memory
// split between the row kernel and the combine).
constexpr int kCombineCols = kCombineBlock;
constexpr int kCombinePairs = SO_COMBINE_PAIRS > 0 ? SO_COMBINE_PAIRS : kGroup;
// Row stride of the stage: the columns of a round, min(c, kCombineCols) (c % 4 == 0).
__host__ __device__ constexpr int64_t combine_stage_width(int64_t c) { return c < kCombineCols ? c : kCombineCols; }
__host__ __device__ constexpr size_t combine_stage_bytes(int64_t c)
{
    return static_cast<size_t>(kCombinePairs) * 2 * static_cast<size_t>(combine_stage_width(c)) * sizeof(float);
}

// Merges the pairs of `run`, in order, at columns col0 + threadIdx.x (one column
// per thread, threads past the row's end idle) into (S, C).  The block copies up
// to kCombinePairs pairs of kCombineCols columns a round into shared memory with
// 16-byte cp.async (through L2, so pairs other blocks stored and released are
// seen), then each thread merges its column.  Every thread of the block calls.
// Needs c % 4 == 0 and a 16-byte aligned partial array.
__device__ __forceinline__ void merge_staged(const float* __restrict__ part, int64_t c, const SlotRun& run,
                                             int64_t col0, float* stage, float& S, float& C)
{
    const int64_t width = (c - col0) < kCombineCols ? (c - col0) : kCombineCols;   // a multiple of 4
    const int quads = static_cast<int>(width / 4);
    const int sw = static_cast<int>(combine_stage_width(c));   // row stride of the stage
    const uint32_t st0 = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
    for (int64_t m0 = 0; m0 < run.cnt; m0 += kCombinePairs) {
        const int k = (run.cnt - m0) < kCombinePairs ? static_cast<int>(run.cnt - m0) : kCombinePairs;
        const int copies = k * 2 * quads;
        for (int e = threadIdx.x; e < copies; e += kCombineBlock) {
            const int pr = e / (2 * quads);
            const int rem = e - pr * 2 * quads;
            const int sc = rem / quads;
            const int q = rem - sc * quads;
            const float* src = part + run.slot(m0 + pr) * 2 * c + sc * c + col0 + 4 * q;
            const uint32_t dst = st0 + static_cast<uint32_t>(((pr * 2 + sc) * sw + 4 * q) * 4);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        if (threadIdx.x < width) {
            for (int r = 0; r < k; ++r) {
                const float xs = stage[(r * 2) * sw + threadIdx.x];
                const float xc = stage[(r * 2 + 1) * sw + threadIdx.x];
                if (m0 + r == 0) {
                    S = xs;
                    C = xc;
                } else {
                    two_sum_merge(S, C, xs, xc);
                }
            }
        }
        __syncthreads();   // the stage is reused by the next round
    }
}

// The same for one column, pairs loaded into registers kCombineIlp at a time
// (any c and alignment).
__device__ __forceinline__ void merge_column(const float* __restrict__ part, int64_t c, const SlotRun& run,
                                             int64_t col, float& S, float& C)
{
    for (int64_t m0 = 0; m0 < run.cnt; m0 += kCombineIlp) {
        float xs[kCombineIlp], xc[kCombineIlp];
#pragma unroll
        for (int r = 0; r < kCombineIlp; ++r) {
            if (m0 + r < run.cnt) {
                const float* q = part + run.slot(m0 + r) * 2 * c + col;
                xs[r] = __ldcg(q);
                xc[r] = __ldcg(q + c);
            }
        }
#pragma unroll
        for (int r = 0; r < kCombineIlp; ++r) {
            if (m0 + r < run.cnt) {
                if (m0 + r == 0) {
                    S = xs[r];
                    C = xc[r];
                } else {
                    two_sum_merge(S, C, xs[r], xc[r]);
                }
            }
        }
    }
}

// The split segments, in one launch: one block per combine group (listed by run
// detection through its head piece), one column per thread.  A segment of one
// group is merged and updated by that block directly; in a longer one every
// block merges its group's partials in piece order into the group head's slot
// and counts the group in its segment (atomic counter; the pair is released
// first), and the block of the last group to arrive merges the groups' pairs in
// group order and applies the update.  The order of every addition is fixed by
// the slots, whichever block arrives last, and no block waits for another.
// Before the wait for the row kernel a block already reads its first group's
// description (run detection's records, complete before the row kernel released
// this grid) and its row's state (a split segment's row is written by this
// kernel alone); only the partials need the row kernel to have finished.
// kStaged: pairs staged through shared memory (c % 4 == 0, aligned partials).
template <class Src, class Epi, bool kStaged>
__global__ void __launch_bounds__(kCombineBlock, 3) k_combine_split(Src src, int64_t c, Epi epi,
                                                                    float* __restrict__ part, int64_t nb,
                                                                    int32_t* d_err)
{
    constexpr int A = Epi::kArrays;
    extern __shared__ float so_combine_stage[];
    __shared__ uint32_t s_arrived;
    const auto merge = [&](const SlotRun& run, int64_t col0, float& S, float& C) {
        if constexpr (kStaged) {
            merge_staged(part, c, run, col0, so_combine_stage, S, C);
        } else {
            if (col0 + threadIdx.x < c) merge_column(part, c, run, col0 + threadIdx.x, S, C);
        }
    };
    struct Group {
        PieceInfo pc;        // the group's head piece
        SlotRun pieces;      // the group's pieces
        SlotRun groups;      // the segment's groups
        int64_t ng;          // groups of the segment
    };
    const auto describe = [&](int64_t t) {
        Group gr;
        gr.pc = src.piece(src.group_index(t));
        int64_t s0, s1;
        src.seg_bounds(gr.pc.u(), s0, s1);
        const SplitSegment seg(s0, s1);
        const int64_t i = seg.index(gr.pc.start);
        const int64_t K = seg.pieces();
        const int64_t next = seg.group_head(seg.group(i) + 1);
        const int64_t cnt = (next < K ? next : K) - i;
        const int64_t g0 = seg.group(0);
        gr.ng = seg.group(K - 1) - g0 + 1;
        // this group's pieces: the first in its own slot, piece p >= 1 of the segment
        // in slot q1/kPieceLen + p - 1; the group heads after the segment's first
        // piece: group g's in slot g*kGroup
        gr.pieces = SlotRun{part_slot(gr.pc.start, nb), seg.q1 / kPieceLen + i - 1, 1, cnt};
        gr.groups = SlotRun{part_slot(s0, nb), g0 * kGroup, kGroup, gr.ng};
        return gr;
    };
    // the row's state at columns col0 + threadIdx.x
    const auto load_row = [&](const PieceInfo& pc, int64_t col0, float (&x)[A][1]) {
        const int64_t col = col0 + threadIdx.x;
        if (col < c) {
#pragma unroll
            for (int a = 0; a < A; ++a)
                if (a < epi.arrays()) x[a][0] = epi.array(a)[epi.base(pc) + col];
        }
    };
    const int64_t G = src.count_groups();
    Group first{};
    float x0[A][1];
    int64_t last0 = 0;
    if (static_cast<int64_t>(blockIdx.x) < G) {
        first = describe(blockIdx.x);
        load_row(first.pc, 0, x0);
        const int64_t* lp = epi.stage_last(first.pc);
        if (lp) last0 = *lp;
    }
    pdl_wait();
    if constexpr (Epi::kEarlyRelease) pdl_release();
    if (read_error(d_err)) return;
    for (int64_t t = blockIdx.x; t < G; t += gridDim.x) {
        const bool is_first = t == static_cast<int64_t>(blockIdx.x);
        const Group gr = is_first ? first : describe(t);
        const PieceInfo& pc = gr.pc;
        const int64_t ng = gr.ng;
        if (ng > 1) {
            if (gr.pieces.cnt > 1) {
                float* pd = part + gr.pieces.first * 2 * c;
                for (int64_t col0 = 0; col0 < c; col0 += kCombineCols) {
                    float S, C;
                    merge(gr.pieces, col0, S, C);
                    const int64_t col = col0 + threadIdx.x;
                    if (col < c) {
                        st_part<1>(pd + col, {S});
                        st_part<1>(pd + c + col, {C});
                    }
                }
            }
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) s_arrived = atomicAdd(src.segment_counter(gr.groups.first), 1u);
            __syncthreads();
            if (static_cast<int64_t>(s_arrived) != ng - 1) continue;   // another group's block finishes it
            __threadfence();
        }
        int64_t last = last0;
        if (!is_first) {
            const int64_t* lp = epi.stage_last(pc);
            last = lp ? *lp : 0;
        }
        const typename Epi::Row row = epi.make_row(pc, last);
        for (int64_t col0 = 0; col0 < c; col0 += kCombineCols) {
            const int64_t col = col0 + threadIdx.x;
            float x[A][1];
            if (is_first && col0 == 0) {
#pragma unroll
                for (int a = 0; a < A; ++a) x[a][0] = x0[a][0];
            } else {
                load_row(pc, col0, x);
            }
            float S, C;
            merge(ng > 1 ? gr.groups : gr.pieces, col0, S, C);
            if (col < c) {
                const float g[1] = {__fadd_rn(S, C)};
                epi.template apply<1>(row, col, x, g);
            }
        }
        __syncthreads();   // every thread has read the row's last_step before it is rewritten
        epi.end_row(row, static_cast<int>(threadIdx.x), kFull);
    }
}

// A small canonical 1-D step (one coordinate per entry, at most kSmallCanon
// entries) in one block and one launch: every entry is checked (index in range,
// strictly ascending, last_step < t) while its state, last_step and gradient are
// read, the block waits at a barrier, and only if the error word is still clear
// is any coordinate written, so the step stays all-or-nothing without a second
// launch.
constexpr int kSmallCanonBlock = 1024;
constexpr int kSmallCanonPer = 4;   // entries a thread
constexpr int64_t kSmallCanon = static_cast<int64_t>(kSmallCanonPer) * kSmallCanonBlock;
static_assert(kSmallCanon == kSmallCanonMax, "the host switch and the kernel agree on the size");
template <class Epi>
__global__ void __launch_bounds__(kSmallCanonBlock) k_small_canon(const int64_t* __restrict__ rows, int64_t n,
                                                                   int64_t r, const float* __restrict__ vals,
                                                                   Epi epi, const int64_t* __restrict__ ls,
                                                                   int64_t t, int32_t* d_err)
{
    constexpr int A = Epi::kArrays;
    pdl_enter();
    PieceInfo pc[kSmallCanonPer];
    float x[kSmallCanonPer][A][1], g[kSmallCanonPer][1];
    int64_t last[kSmallCanonPer];
    bool live[kSmallCanonPer];
#pragma unroll
    for (int j = 0; j < kSmallCanonPer; ++j) {
        const int64_t i = threadIdx.x + static_cast<int64_t>(j) * kSmallCanonBlock;
        live[j] = false;
        if (i >= n) continue;
        const int64_t k = rows[i];
        if (k < 0 || k >= r) {
            set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
            continue;
        }
        if (i > 0 && rows[i - 1] >= k) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
        live[j] = true;
        pc[j].start = static_cast<uint32_t>(i);
        pc[j].end = static_cast<uint32_t>(i + 1);
        pc[j].key = static_cast<uint32_t>(k);
        pc[j].uf = static_cast<uint32_t>(i) & kSingleMask;
        pc[j].perm0 = static_cast<uint32_t>(i);
#pragma unroll
        for (int a = 0; a < A; ++a)
            if (a < epi.arrays()) x[j][a][0] = epi.array(a)[epi.base(pc[j])];
        g[j][0] = vals[i];
        const int64_t* lp = epi.stage_last(pc[j]);
        last[j] = lp ? *lp : 0;
        if (ls && ls[k] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
    }
    __syncthreads();
    if (read_error(d_err)) return;
    const unsigned self = 1u << (threadIdx.x & 31);
#pragma unroll
    for (int j = 0; j < kSmallCanonPer; ++j) {
        if (!live[j]) continue;
        const typename Epi::Row row = epi.make_row(pc[j], last[j]);
        epi.template apply<1>(row, 0, x[j], g[j]);
        epi.end_row(row, 0, self);
    }
}

template <class Epi>
cudaError_t launch_small_canon(const int64_t* rows, int64_t n, int64_t r, const float* vals, const Epi& epi,
                               const int64_t* ls, int64_t t, int32_t* d_err, cudaStream_t s)
{
    SO_PROFILE(Epi::kName, s);
    launch(k_small_canon<Epi>, dim3(1), dim3(kSmallCanonBlock), s, rows, n, r, vals, epi, ls, t, d_err);
    return cudaGetLastError();
}

// ------------------------------------------------------------ launch
template <class K>
int max_blocks(K kernel, int threads, size_t smem = 0)
{
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem);
    return occ > 0 ? occ : 1;
}

// The row kernel, then (on a raw input that may hold split segments) the
// combine kernel.  max_split bounds the number of split segments (0: none).
template <int T, int NV, int V, class Src, class Epi>
cudaError_t launch_shape(const Src& src, int64_t max_pieces, int64_t max_split, const float* vals, int64_t c,
                         const Epi& epi, float* part, int64_t nb, int32_t* d_err, cudaStream_t s)
{
    constexpr int kTeams = kRowBlock / T;
    {
        constexpr size_t smem = long_staged<T, NV, V, Src>() ? long_stage_bytes() : 0;
        static const int occ = [] {
            if (smem > 0) {
                // room for kFusedMinBlocks blocks (plus 1 KB reserved each) of the 228 KB per SM
                const int pct = static_cast<int>(std::min<size_t>(
                    100, (kFusedMinBlocks * (smem + 1024) * 100 + 228 * 1024 - 1) / (228 * 1024)));
                cudaFuncSetAttribute(k_fused_rows<T, NV, V, Src, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem));
                cudaFuncSetAttribute(k_fused_rows<T, NV, V, Src, Epi>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     pct);
            }
            return max_blocks(k_fused_rows<T, NV, V, Src, Epi>, kRowBlock, smem);
        }();
        const int64_t cap = static_cast<int64_t>(occ) * num_sms();
        const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cap, (max_pieces + kTeams - 1) / kTeams)));
        SO_PROFILE(Epi::kName, s);
        launch_smem(k_fused_rows<T, NV, V, Src, Epi>, dim3(blocks), dim3(kRowBlock), smem, s, src, vals, c, epi, part,
                    nb, d_err);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (max_split > 0) {
        SO_PROFILE(Epi::kCombineName, s);
        const int64_t groups = nb + nb / kGroup + 2;   // bound on the combine groups
        if (SO_COMBINE_STAGED && c % 4 == 0 && (reinterpret_cast<uintptr_t>(part) & 15u) == 0) {
            const size_t csmem = combine_stage_bytes(c);
            static int occ_by_quads[kCombineCols / 4 + 1] = {};   // occupancy by stage width, looked up once
            int& occ = occ_by_quads[combine_stage_width(c) / 4];
            if (occ == 0) {
                // the largest stage any row width takes (the attribute belongs to the kernel, whose
                // launches for narrower rows ask for less)
                cudaFuncSetAttribute(k_combine_split<Src, Epi, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(combine_stage_bytes(kCombineCols)));
                occ = max_blocks(k_combine_split<Src, Epi, true>, kCombineBlock, csmem);
            }
            const int64_t gb = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(occ) * num_sms(), groups));
            launch_smem(k_combine_split<Src, Epi, true>, dim3(static_cast<unsigned>(gb)), dim3(kCombineBlock), csmem,
                        s, src, c, epi, part, nb, d_err);
        } else {
            static const int occ = max_blocks(k_combine_split<Src, Epi, false>, kCombineBlock);
            const int64_t gb = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(occ) * num_sms(), groups));
            launch(k_combine_split<Src, Epi, false>, dim3(static_cast<unsigned>(gb)), dim3(kCombineBlock), s, src, c,
                   epi, part, nb, d_err);
        }
        return cudaGetLastError();
    }
    return cudaSuccess;
}

// Team shape: smallest power-of-two team that covers a row with one vector per
// lane; rows wider than 32 vectors give each lane 2 vectors per chunk and are
// walked in chunks of 256 (or 128 scalar) columns.
template <class Src, class Epi>
cudaError_t launch_fused(const Src& src, int64_t max_pieces, int64_t max_split, const float* vals, int64_t c,
                         const Epi& epi, float* part, int64_t nb, int vec4, int32_t* d_err, cudaStream_t s)
{
    if (max_pieces <= 0) return cudaSuccess;
#define SO_LAUNCH(T, NV, V) \
    launch_shape<T, NV, V>(src, max_pieces, max_split, vals, c, epi, part, nb, d_err, s)
    if (vec4) {
        const int64_t nv = c / 4;
        if (nv <= 1) return SO_LAUNCH(1, 1, 4);
        if (nv <= 2) return SO_LAUNCH(2, 1, 4);
        if (nv <= 4) return SO_LAUNCH(4, 1, 4);
        if (nv <= 8) return SO_LAUNCH(8, 1, 4);
        if (nv <= 16) return SO_LAUNCH(16, 1, 4);
        if (nv <= 32) return SO_LAUNCH(32, 1, 4);
        return SO_LAUNCH(32, 2, 4);   // wider rows: chunks of 256 columns
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
    return SortedSrc{ws.rec, ws.vals[ws.final_buf], ws.seg_off, ws.mlist, ws.slist, ws.glist, ws.counts, ws.scnt};
}

}  // namespace so
