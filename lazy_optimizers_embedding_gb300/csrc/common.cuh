// common.cuh -- device helpers and internal launch interfaces shared by the
// translation units of libsparseopt (sm_103a).
#pragma once

#include <utility>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "sparseopt.h"

namespace so {

// ---------------------------------------------------------------- launches
// Every kernel of this library is launched with programmatic dependent launch
// allowed.  A kernel waits (griddepcontrol.wait) until the previous kernel on
// the stream has completed and its memory is visible before it touches memory
// another kernel uses; the histogram kernel alone first counts the caller's
// index array.  Then it lets the next kernel's blocks be scheduled
// (griddepcontrol.launch_dependents), so that the next grid is resident when
// this one completes.  A kernel that writes an output the caller may pass as
// the index array of the next call (canonical indices, offsets, permutation,
// linear indices, converted structures, gathered or summed values) skips that
// early release: its dependents start only once all its blocks have exited, so
// the histogram kernel's early read of an index array never precedes the write.
// Results and stream order are those of plain launches.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_release();
}

template <class... P, class... A>
inline cudaError_t launch(void (*kernel)(P...), dim3 grid, dim3 block, cudaStream_t s, A&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// The same with dynamic shared memory.
template <class... P, class... A>
inline cudaError_t launch_smem(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               A&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}


constexpr unsigned kFull = 0xffffffffu;
constexpr int kBlock = 256;            // threads per block of every kernel here
#ifndef SO_PIECE_LEN
#define SO_PIECE_LEN 32
#endif
constexpr int kPieceLen = SO_PIECE_LEN;   // L: sorted entries summed by one team before a partial
// Keys per thread of a radix pass and sorted warp rows per thread of run
// detection (at most 21): kSortItems / kRunItems below kLargeN
// entries, the large-input sizes from kLargeN on (fewer, larger tiles shorten the
// look-back chains of large inputs; smaller tiles start more blocks on small ones).
#ifndef SO_SORT_ITEMS
#define SO_SORT_ITEMS 8
#endif
#ifndef SO_RUN_ITEMS
#define SO_RUN_ITEMS 8
#endif
#ifndef SO_SORT_ITEMS_LARGE
#define SO_SORT_ITEMS_LARGE 16
#endif
#ifndef SO_RUN_ITEMS_LARGE
#define SO_RUN_ITEMS_LARGE 16
#endif
#ifndef SO_LARGE_N
#define SO_LARGE_N (1 << 19)
#endif
constexpr int kSortItems = SO_SORT_ITEMS;
constexpr int kRunItems = SO_RUN_ITEMS;
constexpr int kSortItemsLarge = SO_SORT_ITEMS_LARGE;
constexpr int kRunItemsLarge = SO_RUN_ITEMS_LARGE;
constexpr int64_t kLargeN = SO_LARGE_N;
constexpr int kMaxPasses = 4;          // 8-bit digits, keys < 2^32
#ifndef SO_GROUP
#define SO_GROUP 16
#endif
constexpr int kGroup = SO_GROUP;       // pieces of a split segment merged by one combine block first
constexpr int kHistItems = 8;          // keys a histogram thread requests at once
#ifndef SO_HIST_BLOCKS
#define SO_HIST_BLOCKS 256
#endif
#ifndef SO_HIST_KEYS
#define SO_HIST_KEYS 8192
#endif
// Partial pairs a combine block stages per round (0: a group's worth).
#ifndef SO_COMBINE_PAIRS
#define SO_COMBINE_PAIRS 0
#endif
#ifndef SO_RADIX_LOOK
#define SO_RADIX_LOOK 16
#endif
constexpr int kMaxHistBlocks = SO_HIST_BLOCKS;     // histogram blocks at most
constexpr int kHistKeysPerBlock = SO_HIST_KEYS;    // keys per histogram block (fewer blocks for small n)
constexpr int kHistPrefetch = 32;                  // block counts a first-pass thread requests with its keys
constexpr int kRadixLook = SO_RADIX_LOOK;          // predecessor tiles a radix look-back reads per round trip
constexpr uint32_t kSingleMask = 0x3fffffffu;   // segment index bits of a piece record
constexpr uint32_t kMultiFlag = 0x80000000u;    // piece of a segment split into several pieces
constexpr uint32_t kLongFlag = 0x40000000u;     // whole segment of more than kShortLen entries
// Pieces of at most kShortLen entries are the row kernel's short pieces; longer
// ones (and all pieces of split segments) its long pieces, worked first.
#ifndef SO_SHORT_LEN
#define SO_SHORT_LEN 4
#endif
constexpr int kShortLen = SO_SHORT_LEN;
// Bounded waits on another block's published value: after this many polls the
// waiting block records SPARSE_ERR_INTERNAL and carries on with a zero value.
constexpr uint32_t kSpinLimit = 1u << 22;

// ------------------------------------------------------------------ errors
__device__ __forceinline__ void set_error(int32_t* d_err, int code)
{
    atomicCAS(d_err, 0, code);
}

__device__ __forceinline__ int read_error(const int32_t* d_err)
{
    return *reinterpret_cast<const volatile int32_t*>(d_err);
}

// ------------------------------------------------------- relaxed gpu-scope I/O
__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p)
{
    return *reinterpret_cast<const volatile uint32_t*>(p);
}
__device__ __forceinline__ unsigned long long ld_volatile(const unsigned long long* p)
{
    return *reinterpret_cast<const volatile unsigned long long*>(p);
}
__device__ __forceinline__ void st_volatile(uint32_t* p, uint32_t v)
{
    *reinterpret_cast<volatile uint32_t*>(p) = v;
}
__device__ __forceinline__ void st_volatile(unsigned long long* p, unsigned long long v)
{
    *reinterpret_cast<volatile unsigned long long*>(p) = v;
}

// ------------------------------------------------- error-free transformation
// Knuth's TwoSum: s + x = t + e exactly, t = fl(s + x).  Rounding-mode explicit
// intrinsics keep the compiler from contracting or reassociating.
__device__ __forceinline__ void two_sum_acc(float& s, float& c, float x)
{
    const float t = __fadd_rn(s, x);
    const float bp = __fsub_rn(t, s);
    const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(x, bp));
    s = t;
    c = __fadd_rn(c, e);
}

// (s, c) += (s2, c2), both compensated pairs.
__device__ __forceinline__ void two_sum_merge(float& s, float& c, float s2, float c2)
{
    two_sum_acc(s, c, s2);
    c = __fadd_rn(c, c2);
}

// --------------------------------------------------------------- warp scans
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t x, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, x, d);
        if (lane >= d) x += y;
    }
    return x;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x)
{
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(kFull, x, d);
    return x;
}

// Exclusive scan of one uint32 per thread over a kBlock-thread block.
// `tmp` is shared scratch of kBlock/32 + 1 words.  Returns the exclusive
// prefix; *total receives the block sum.  Every thread of the block must call.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t x, uint32_t* tmp, uint32_t* total)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_scan(x, lane);
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kBlock / 32 ? tmp[lane] : 0u;
        const uint32_t wi = warp_incl_scan(w, lane);
        if (lane < kBlock / 32) tmp[lane] = wi - w;
        if (lane == kBlock / 32 - 1) tmp[kBlock / 32] = wi;
    }
    __syncthreads();
    const uint32_t res = tmp[warp] + incl - x;
    *total = tmp[kBlock / 32];
    __syncthreads();
    return res;
}

// ------------------------------------------------------------ workspace map
struct WsLayout {
    int64_t n, c, nb;
    int passes, sort_items, run_items, sort_tiles, run_tiles, hist_blocks;
    size_t keys0, keys1, vals0, vals1, rec, seg_off, mlist, slist, glist, part, bh, gh;
    size_t ctrl_begin, counts, rstatus, dstatus, scnt, ctrl_end;
    size_t total;
};

// counts[] word indices
enum { kCtrPass0 = 1, kCtrRun = 5, kCntU = 8, kCntP = 9, kCntM = 10, kCntS = 11, kCntG = 12, kTicketS = 14,
       kCountsWords = 16 };

WsLayout ws_layout(int64_t n, int64_t c, int64_t bound);

// Device pointers carved out of a workspace.
struct SortWs {
    uint32_t* keys[2];
    uint32_t* vals[2];
    uint4* rec;           // [P+1] piece records {start, key, u | multi, perm of start}
    uint32_t* seg_off;    // [U+1]
    uint32_t* mlist;      // [M] indices of the long pieces (any order)
    uint32_t* slist;      // [S] indices of the first pieces of split segments (any order)
    uint32_t* glist;      // [G] indices of the pieces heading a combine group (any order)
    float* part;          // partial sums: [2*nb slots][2][c]
    uint32_t* bh;         // [hist_blocks][4][256] digit histograms, one set per block
    uint32_t* gh;         // [4][256] whole-input digit histograms of the later passes
    uint32_t* counts;     // [16]: tile counters, U, P, M, S, G, the short pieces' ticket counter
    uint32_t* rstatus;    // [passes][sort_tiles][256]
    unsigned long long* dstatus;  // [run_tiles]
    uint32_t* scnt;       // [2*nb] groups merged per split segment (zeroed with the control block)
    int final_buf;        // which keys/vals buffer holds the sorted result
};

SortWs carve(const WsLayout& L, void* ws);

// ------------------------------------------------------------ launch helpers
int num_sms();

// Sorts the keys (uint32 of idx) stably with their positions and detects runs.
// Afterwards: ws.rec / ws.seg_off / counts[kCntU], counts[kCntP] describe the
// segments; optional int64 outputs (idx_out, seg_off_out, perm_out, d_nnz_out)
// are filled for sparse_canonicalize.  When ls != nullptr, each unique key k
// (a row) is checked for ls[k] < t (per row) or ls[k*c + j] < t (per coord).
cudaError_t sort_and_segment(const int64_t* idx, int64_t n, int64_t c, int64_t bound,
                             const WsLayout& L, SortWs& ws, int64_t* idx_out,
                             int64_t* seg_off_out, int64_t* perm_out, int64_t* d_nnz_out,
                             const int64_t* ls, int ls_per_coord, int64_t t, int32_t* d_err,
                             cudaStream_t s);

// Checks a canonical row-COO: 0 <= rows[i] < r, strictly ascending, last_step < t.
cudaError_t check_canonical_rows(const int64_t* rows, int64_t n, int64_t r, int64_t c,
                                 const int64_t* ls, int ls_per_coord, int64_t t,
                                 int32_t* d_err, cudaStream_t s);

// ------------------------------------------------------- update parameters
struct AdamParams {
    float* p;
    float* m;
    float* v;
    int64_t* ls;
    int ls_per_coord;
    int dd;               // DormancyDecay
    int64_t t;
    float beta1, beta2;   // decay factors
    float omb1, omb2;     // 1 - beta
    float log2b1, log2b2; // log2(beta) (-inf for beta = 0)
    float inv_bc1, inv_bc2;  // 1 / (1 - beta^t)
    float lr, eps;
    float wd, wd_lo;      // weight decay as hi + lo (0: none)
    int wd_decoupled;     // 1: added to the descent direction (AdamW); 0: to the gradient (L2)
};

struct SgdParams {
    float* p;
    float* buf;
    float lr;
    float momentum, momentum_lo;  // momentum = momentum + momentum_lo (double split into two floats)
    float wd, wd_lo;              // weight decay, split the same way
};

struct StoreParams {
    float* out;           // [U][c]
};

// Row-fused update from sorted segments (raw input) or canonical rows.
cudaError_t fused_rows_adam_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                   const AdamParams& P, int vec4, int32_t* d_err, cudaStream_t s);
cudaError_t fused_rows_adam_canon(const int64_t* rows, int64_t n, const float* vals, int64_t c,
                                  const AdamParams& P, int vec4, int32_t* d_err, cudaStream_t s);
cudaError_t fused_rows_sgd_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                  const SgdParams& P, int vec4, int32_t* d_err, cudaStream_t s);
cudaError_t fused_rows_sgd_canon(const int64_t* rows, int64_t n, const float* vals, int64_t c,
                                 const SgdParams& P, int vec4, int32_t* d_err, cudaStream_t s);
cudaError_t fused_rows_store_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                    const StoreParams& P, int vec4, int32_t* d_err, cudaStream_t s);
// A canonical 1-D SGD step (c == 1) of at most 4,096 entries: check and update in
// one single-block launch (for Adam the check and the row kernel as two launches
// measured as fast or faster, so Adam keeps them).
constexpr int64_t kSmallCanonMax = 4096;
cudaError_t small_canon_sgd(const int64_t* rows, int64_t n, int64_t r, const float* vals, const SgdParams& P,
                            int32_t* d_err, cudaStream_t s);

// CSR (element-granular) paths.
// rows_list (full_rows only, may be NULL): filled with the listed rows; ent_row /
// ent_gap (not full_rows, may be NULL): every entry's row and gap; see k_csr_check.
cudaError_t csr_check(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                      int full_rows, const int64_t* ls, int ls_per_coord, int64_t t, int64_t* rows_list,
                      int32_t* ent_row, int32_t* ent_gap, int32_t* d_err, cudaStream_t s);
// Element-granular CSR updates from the check's per-entry rows (and gaps).
cudaError_t csr_adam_flat(const int32_t* cols, const float* vals, const int32_t* ent_row, const int32_t* ent_gap,
                          int64_t c, int64_t nnz, const AdamParams& P, int32_t* d_err, cudaStream_t s);
cudaError_t csr_sgd_flat(const int32_t* cols, const float* vals, const int32_t* ent_row, int64_t c, int64_t nnz,
                         const SgdParams& P, int32_t* d_err, cudaStream_t s);
cudaError_t read_rows(const float* table, int64_t r, int64_t c, const int64_t* idx, int64_t n, float* out, int vec4,
                      int32_t* d_err, cudaStream_t s);
cudaError_t check_finite(const float* vals, int64_t n, int32_t* d_err, cudaStream_t s);
cudaError_t check_state_rows(const float* m, const float* v, int64_t r, int64_t c, const int64_t* idx, int64_t n,
                             int vec4, int32_t* d_err, cudaStream_t s);
cudaError_t check_state_csr(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c, int64_t nnz,
                            const float* m, const float* v, int32_t* d_err, cudaStream_t s);
cudaError_t csr_adam(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r,
                     int64_t c, int64_t nnz, const AdamParams& P, int32_t* d_err, cudaStream_t s);
cudaError_t csr_sgd(const int64_t* row_off, const int32_t* cols, const float* vals, int64_t r,
                    int64_t c, int64_t nnz, const SgdParams& P, int32_t* d_err, cudaStream_t s);
cudaError_t csr_to_coo(const int64_t* row_off, const int32_t* cols, int64_t r, int64_t c,
                       int64_t nnz, int64_t* lin_out, int32_t* d_err, cudaStream_t s);
cudaError_t coo_to_csr(const int64_t* lin, int64_t nnz, int64_t r, int64_t c, int64_t* row_off_out,
                       int32_t* cols_out, int32_t* d_err, cudaStream_t s);
cudaError_t row_coo_to_csr(const int64_t* rows, int64_t nrows, int64_t r, int64_t c,
                           int64_t* row_off_out, int32_t* cols_out, int32_t* d_err, cudaStream_t s);

}  // namespace so
