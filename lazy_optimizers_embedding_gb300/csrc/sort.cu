// sort.cu -- canonicalisation front half on the device:
//   K1 range check + digit histograms of every radix pass,
//   K2 stable LSD radix sort of (key, position), one 8-bit digit per pass,
//      single-sweep per pass with decoupled look-back between tiles,
//   K3 run detection: segment heads (key changes) and piece heads (segment heads
//      plus every kPieceLen-th sorted position), compacted by a block scan with
//      decoupled look-back.
// Canonical form per "Module sparse_optimizer" (optirs-gpu 0.3.2 docs),
// "Sparse gradient representations" (strictly ascending indices); sorting and
// duplicate detection per the "DiskSparseAdam (DSA)" README, "Safe Duplicate
// Aggregation & Sorted I/O".
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "profile.cuh"

namespace so {

int num_sms()
{
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    return sms;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int key_bits(int64_t bound)
{
    int b = 1;
    while (b < 32 && (int64_t(1) << b) < bound) ++b;
    return b;
}

WsLayout ws_layout(int64_t n, int64_t c, int64_t bound)
{
    WsLayout L{};
    if (n < 1) n = 1;
    if (c < 1) c = 1;
    L.n = n;
    L.c = c;
    L.nb = (n + kPieceLen - 1) / kPieceLen;
    L.passes = (key_bits(bound) + 7) / 8;
    L.sort_items = n >= kLargeN ? kSortItemsLarge : kSortItems;
    L.run_items = n >= kLargeN ? kRunItemsLarge : kRunItems;
    L.sort_tiles = (int)((n + kBlock * L.sort_items - 1) / (kBlock * L.sort_items));
    L.run_tiles = (int)((n + kBlock * L.run_items - 1) / (kBlock * L.run_items));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = align_up(off, 256);
        size_t at = off;
        off += bytes;
        return at;
    };
    L.keys0 = take(sizeof(uint32_t) * n);
    L.keys1 = take(sizeof(uint32_t) * n);
    L.vals0 = take(sizeof(uint32_t) * n);
    L.vals1 = take(sizeof(uint32_t) * n);
    L.rec = take(sizeof(uint4) * (size_t)(n + L.nb + 2));
    L.seg_off = take(sizeof(uint32_t) * (size_t)(n + 1));
    L.mlist = take(sizeof(uint32_t) * (size_t)(n + L.nb + 2));
    L.slist = take(sizeof(uint32_t) * (size_t)(L.nb + 1));
    L.glist = take(sizeof(uint32_t) * (size_t)(L.nb + n / (kPieceLen * kGroup) + 2));
    L.part = take(sizeof(float) * (size_t)(2 * L.nb) * 2 * (size_t)c);
    L.hist_blocks = (int)std::min<int64_t>((n + kHistKeysPerBlock - 1) / kHistKeysPerBlock, kMaxHistBlocks);
    L.bh = take(sizeof(uint32_t) * (size_t)L.hist_blocks * kMaxPasses * 256);
    L.gh = take(sizeof(uint32_t) * kMaxPasses * 256);
    off = align_up(off, 256);
    L.ctrl_begin = off;
    L.counts = take(sizeof(uint32_t) * kCountsWords);
    L.rstatus = take(sizeof(uint32_t) * (size_t)L.passes * L.sort_tiles * 256);
    L.dstatus = take(sizeof(unsigned long long) * (size_t)L.run_tiles);
    L.scnt = take(sizeof(uint32_t) * (size_t)(2 * L.nb));
    L.ctrl_end = align_up(off, 256);
    L.total = L.ctrl_end;
    return L;
}

SortWs carve(const WsLayout& L, void* ws)
{
    char* b = static_cast<char*>(ws);
    SortWs w{};
    w.keys[0] = reinterpret_cast<uint32_t*>(b + L.keys0);
    w.keys[1] = reinterpret_cast<uint32_t*>(b + L.keys1);
    w.vals[0] = reinterpret_cast<uint32_t*>(b + L.vals0);
    w.vals[1] = reinterpret_cast<uint32_t*>(b + L.vals1);
    w.rec = reinterpret_cast<uint4*>(b + L.rec);
    w.seg_off = reinterpret_cast<uint32_t*>(b + L.seg_off);
    w.mlist = reinterpret_cast<uint32_t*>(b + L.mlist);
    w.slist = reinterpret_cast<uint32_t*>(b + L.slist);
    w.glist = reinterpret_cast<uint32_t*>(b + L.glist);
    w.part = reinterpret_cast<float*>(b + L.part);
    w.bh = reinterpret_cast<uint32_t*>(b + L.bh);
    w.gh = reinterpret_cast<uint32_t*>(b + L.gh);
    w.counts = reinterpret_cast<uint32_t*>(b + L.counts);
    w.rstatus = reinterpret_cast<uint32_t*>(b + L.rstatus);
    w.dstatus = reinterpret_cast<unsigned long long*>(b + L.dstatus);
    w.scnt = reinterpret_cast<uint32_t*>(b + L.scnt);
    w.final_buf = (L.passes - 1) & 1;
    return w;
}

// ---------------------------------------------------------------------- K1
// Range check (0 <= idx < bound) and the digit histograms of all passes, one
// set per block (bh[block][pass][digit], read by every radix tile), so nothing
// has to be zeroed before this kernel: it zeroes the control words the later
// kernels of the call count in (ctrl, 16-byte words).  Every key is counted,
// valid or not, with the same truncation the radix passes use, so the scatter
// offsets stay inside [0, n) whatever the input.  Each thread requests its
// kHistItems keys at once (128-bit loads when aligned), then counts them in
// shared memory.
__global__ void __launch_bounds__(kBlock) k_range_hist(const int64_t* __restrict__ idx, uint32_t n,
                                                       int64_t bound, int passes, uint32_t* __restrict__ bh,
                                                       uint4* __restrict__ ctrl, uint32_t ctrl_words,
                                                       int32_t* d_err)
{
    // Counting reads only the caller's index array and shared memory, so it runs
    // before the wait for the previous kernel on the stream (which may still be
    // using the workspace); the control words and the histograms are written
    // after it.
    __shared__ uint32_t sh[kMaxPasses * 256];
    for (int i = threadIdx.x; i < kMaxPasses * 256; i += kBlock) sh[i] = 0;
    __syncthreads();
    int bad = 0;
    const uint32_t stride = gridDim.x * kBlock * kHistItems;
    for (uint32_t i0 = (blockIdx.x * kBlock + threadIdx.x) * kHistItems; i0 < n; i0 += stride) {
        int64_t k[kHistItems];
        if (i0 + kHistItems <= n && (reinterpret_cast<uintptr_t>(idx + i0) & 15u) == 0) {
#pragma unroll
            for (int j = 0; j < kHistItems; j += 2) {
                const longlong2 q = *reinterpret_cast<const longlong2*>(idx + i0 + j);
                k[j] = q.x;
                k[j + 1] = q.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kHistItems; ++j) k[j] = (i0 + j < n) ? idx[i0 + j] : 0;
        }
#pragma unroll
        for (int j = 0; j < kHistItems; ++j) {
            if (i0 + j < n) {
                bad |= (k[j] < 0) | (k[j] >= bound);
                const uint32_t key = static_cast<uint32_t>(static_cast<uint64_t>(k[j]));
                for (int p = 0; p < passes; ++p) atomicAdd(&sh[p * 256 + ((key >> (8 * p)) & 255u)], 1u);
            }
        }
    }
    const int any_bad = __syncthreads_or(bad);
    pdl_enter();
    for (uint32_t i = blockIdx.x * kBlock + threadIdx.x; i < ctrl_words; i += gridDim.x * kBlock)
        ctrl[i] = make_uint4(0u, 0u, 0u, 0u);
    if (any_bad && threadIdx.x == 0) set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
    uint32_t* mine = bh + static_cast<size_t>(blockIdx.x) * kMaxPasses * 256;
    for (int i = threadIdx.x; i < passes * 256; i += kBlock) mine[i] = sh[i];
}

// Sum over histogram blocks b0 .. hb-1 of one digit's count (32 loads in flight).
__device__ __forceinline__ uint32_t sum_hist(const uint32_t* __restrict__ bh, int b0, int hb, int digit)
{
    uint32_t s = 0;
    for (int b = b0; b < hb; b += 32) {
        uint32_t h[32];
#pragma unroll
        for (int q = 0; q < 32; ++q)
            h[q] = (b + q < hb) ? bh[static_cast<size_t>(b + q) * kMaxPasses * 256 + digit] : 0u;
#pragma unroll
        for (int q = 0; q < 32; ++q) s += h[q];
    }
    return s;
}

// ---------------------------------------------------------------------- K2
// One stable counting pass over digit (key >> shift) & 255.  Tiles are taken in
// launch order from an atomic counter, so a tile only ever waits on tiles that
// are already running.  Per tile:
//   1. warp-level ranking: the lanes holding a digit are found by each lane
//      OR-ing its bit into a per-warp shared word of its digit (a fixed cost,
//      where a match instruction's grows with the distinct digits in the warp);
//      warp w owns a contiguous run of the tile, items in order, so ranks are
//      stable;
//   2. per-digit tile counts are published (flag 1 = aggregate), the exclusive
//      prefix over earlier tiles is found by look-back and republished
//      (flag 2 = inclusive); status word = count << 2 | flag;
//   3. the tile is reordered by digit in shared memory and written out, each
//      digit's run landing contiguously at its global offset.
template <bool kFirst, int SI>
__global__ void __launch_bounds__(kBlock, 2) k_radix_pass(const int64_t* __restrict__ idx64,
                                                       const uint32_t* __restrict__ kin,
                                                       const uint32_t* __restrict__ vin,
                                                       uint32_t* __restrict__ kout,
                                                       uint32_t* __restrict__ vout, uint32_t n, int shift,
                                                       const uint32_t* __restrict__ bh, int hist_blocks,
                                                       uint32_t* __restrict__ gh, int passes,
                                                       uint32_t* status, uint32_t* tile_ctr,
                                                       int32_t* d_err)
{
    constexpr int kWarps = kBlock / 32;
    __shared__ uint32_t s_wh[kWarps][256];
    __shared__ uint32_t s_gbase[256];
    __shared__ uint32_t s_texcl[256];
    __shared__ uint32_t s_scan[kWarps + 1];
    __shared__ uint32_t s_keys[(kBlock * SI)];
    __shared__ uint32_t s_vals[(kBlock * SI)];
    __shared__ uint32_t s_tile;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    // the tile counters were zeroed by the histogram kernel, which has completed
    // before any later pass can start (each pass waits on its predecessor before
    // releasing its dependents): passes after the first take their tile before
    // the wait
    if (!kFirst && tid == 0) s_tile = atomicAdd(tile_ctr, 1u);
    for (int i = tid; i < kWarps * 256; i += kBlock) (&s_wh[0][0])[i] = 0u;
    pdl_enter();
    if (kFirst && tid == 0) s_tile = atomicAdd(tile_ctr, 1u);
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint32_t base = tile * (kBlock * SI);
    const uint32_t tile_n = min(static_cast<uint32_t>((kBlock * SI)), n - base);

    // digit tid over the whole input.  The first pass sums the histogram blocks'
    // counts (the first kHistPrefetch requested together with the tile's keys)
    // and tile t also writes the global histograms of passes 1 + t, 1 + t + tiles,
    // ... for the later passes, which read them with one load.
    uint32_t hcount[kHistPrefetch];
    if (kFirst) {
#pragma unroll
        for (int q = 0; q < kHistPrefetch; ++q)
            hcount[q] = (q < hist_blocks) ? bh[static_cast<size_t>(q) * kMaxPasses * 256 + tid] : 0u;
    } else {
        hcount[0] = gh[tid];
    }
    uint32_t key[SI], val[SI], rank[SI];
    int dig[SI];
#pragma unroll
    for (int i = 0; i < SI; ++i) {
        const uint32_t local = warp * 32 * SI + i * 32 + lane;
        const bool valid = local < tile_n;
        uint32_t k = 0, v = 0;
        if (valid) {
            const uint32_t pos = base + local;
            if (kFirst) {
                k = static_cast<uint32_t>(static_cast<uint64_t>(idx64[pos]));
                v = pos;
            } else {
                k = kin[pos];
                v = vin[pos];
            }
        }
        key[i] = k;
        val[i] = v;
        dig[i] = valid ? static_cast<int>((k >> shift) & 255u) : 256;
    }
    const uint32_t lt = (1u << lane) - 1u;
    __shared__ uint32_t s_match[kWarps][256];
    for (int i = lane; i < 256; i += 32) s_match[warp][i] = 0u;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < SI; ++i) {
        const int d = dig[i];
        if (d < 256) atomicOr(&s_match[warp][d], 1u << lane);
        __syncwarp();
        const uint32_t peers = d < 256 ? s_match[warp][d] : 0u;
        uint32_t b = 0;
        if (d < 256) b = s_wh[warp][d];
        __syncwarp();
        if (d < 256 && lane == __ffs(peers) - 1) {
            s_wh[warp][d] = b + __popc(peers);
            s_match[warp][d] = 0u;
        }
        __syncwarp();
        rank[i] = b + __popc(peers & lt);
    }
    __syncthreads();

    // thread tid owns digit tid
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t cnt = s_wh[w][tid];
        s_wh[w][tid] = run;
        run += cnt;
    }
    const uint32_t tcount = run;
    uint32_t* my = status + static_cast<size_t>(tile) * 256 + tid;
    st_volatile(my, (tcount << 2) | (tile == 0 ? 2u : 1u));

    uint32_t total;
    s_texcl[tid] = block_excl_scan(tcount, s_scan, &total);
    uint32_t gcount = 0;
    if (kFirst) {
#pragma unroll
        for (int q = 0; q < kHistPrefetch; ++q) gcount += hcount[q];
        gcount += sum_hist(bh, kHistPrefetch, hist_blocks, tid);
        for (int p = 1 + static_cast<int>(tile); p < passes; p += static_cast<int>(gridDim.x))
            gh[p * 256 + tid] = sum_hist(bh + p * 256, 0, hist_blocks, tid);
    } else {
        gcount = hcount[0];
    }
    const uint32_t gexcl = block_excl_scan(gcount, s_scan, &total);

    // look-back: kLook predecessor words per round trip, consumed nearest first
    // until an inclusive one; a word not yet published stops the round (its
    // tile started earlier, so it publishes soon) and is read again.
    constexpr int kLook = kRadixLook;
    uint32_t excl = 0;
    if (tile > 0) {
        int64_t j = static_cast<int64_t>(tile) - 1;
        uint32_t spins = 0;
        bool done = false;
        while (!done && j >= 0) {
            uint32_t w[kLook];
#pragma unroll
            for (int q = 0; q < kLook; ++q)
                w[q] = (j - q >= 0) ? ld_volatile(status + static_cast<size_t>(j - q) * 256 + tid) : 2u;
            int used = 0;
#pragma unroll
            for (int q = 0; q < kLook; ++q) {
                if (done || used < q) break;
                const uint32_t flag = w[q] & 3u;
                if (flag == 0u) break;
                excl += w[q] >> 2;
                ++used;
                if (flag == 2u) done = true;
            }
            if (done) break;
            if (used == 0) {
                if (++spins > kSpinLimit) {
                    set_error(d_err, SPARSE_ERR_INTERNAL);
                    break;
                }
                if (spins > 64) __nanosleep(64);
                continue;
            }
            j -= used;
        }
        st_volatile(my, ((excl + tcount) << 2) | 2u);
    }
    s_gbase[tid] = gexcl + excl;
    __syncthreads();

#pragma unroll
    for (int i = 0; i < SI; ++i) {
        const int d = dig[i];
        if (d < 256) {
            const uint32_t lp = s_texcl[d] + s_wh[warp][d] + rank[i];
            s_keys[lp] = key[i];
            s_vals[lp] = val[i];
        }
    }
    __syncthreads();
    for (uint32_t i = tid; i < tile_n; i += kBlock) {
        const uint32_t k = s_keys[i];
        const uint32_t d = (k >> shift) & 255u;
        const uint32_t dst = s_gbase[d] + (i - s_texcl[d]);
        kout[dst] = k;
        vout[dst] = s_vals[i];
    }
}

// ---------------------------------------------------------------------- K3
// Run detection over the sorted keys.  Position q is a segment head when it is
// the first position or its key differs from the previous one.  It is a piece
// head when it is a segment head, or when q is a multiple of kPieceLen and
// position q - kPieceLen belongs to the same segment.  So a segment of at most
// kPieceLen entries is always one piece (wherever it lies), and a longer one is
// cut at the multiples of kPieceLen that lie at least kPieceLen past its start:
// its first piece holds kPieceLen .. 2*kPieceLen-1 entries, the others at most
// kPieceLen.  Outputs (u = segment index,
// j = piece index):
//   seg_off[u] = first sorted position of segment u, seg_off[U] = n
//   rec[j] = {start, key, u | kMultiFlag if the segment spans several pieces
//             | kLongFlag if it is one piece of more than kShortLen entries,
//             input position of the start}, rec[P] = {n, 0, 0, 0}
//   mlist[0 .. M) = the indices j of the flagged pieces, and
//   slist[0 .. S) = the indices j of the first pieces of split segments,
//   glist[0 .. G) = the indices j of the pieces that head a combine group: the
//             first piece of a split segment, and a later piece of one that
//             starts at a multiple of kPieceLen*kGroup,
//             each in no particular order (appended through atomic counters,
//             one per list and warp; the order in which they are processed
//             does not affect any result)
// Status word of a tile: flag << 62 | heads << 31 | pieces.
template <int RI>
__global__ void __launch_bounds__(kBlock) k_run_detect(
    const uint32_t* __restrict__ skey, const uint32_t* __restrict__ sperm, uint32_t n,
    uint4* __restrict__ rec, uint32_t* __restrict__ seg_off, uint32_t* __restrict__ mlist,
    uint32_t* __restrict__ slist, uint32_t* __restrict__ glist,
    unsigned long long* dstatus,
    uint32_t* tile_ctr, uint32_t* counts, int64_t* __restrict__ idx_out,
    int64_t* __restrict__ seg_off_out, int64_t* __restrict__ perm_out, int64_t* d_nnz_out,
    const int64_t* __restrict__ ls, int ls_per_coord, int64_t c, int64_t bound, int64_t t,
    int32_t* d_err)
{
    // Warp-striped: warp w of tile T owns the 32*RI sorted positions from
    // wbase = (T*kWarps + w)*32*RI, row i of them in item i (lane l holds
    // position wbase + 32 i + l), so every load and store of a row is one
    // coalesced warp access; neighbours come from shuffles, and positions are
    // counted in order by ballots.  Piece boundaries (multiples of kPieceLen)
    // are lane 0 of a row.
    static_assert(kPieceLen == 32, "piece boundaries are lane 0 of a warp row");
    static_assert(kShortLen > 0 && kShortLen < 32, "a long segment's test key lies in the next row at most");
    static_assert(3 * RI <= 64, "kinds holds 3 bits per item");
    constexpr unsigned long long kValMask = (1ull << 62) - 1ull;
    constexpr int kWarps = kBlock / 32;
    __shared__ uint32_t s_warp[kWarps];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_tile;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    // the tile counter was zeroed by the histogram kernel, complete before the
    // radix passes released this grid: the tile is taken before the wait
    if (tid == 0) s_tile = atomicAdd(tile_ctr, 1u);
    pdl_wait();
    // canonical outputs are caller memory the next call may read as its index
    // array: with any of them requested, dependents start after this grid exits
    if (idx_out == nullptr && seg_off_out == nullptr && perm_out == nullptr && d_nnz_out == nullptr) pdl_release();
    __syncthreads();
    const uint32_t tile = s_tile;
    const uint32_t wbase = (tile * kWarps + warp) * (32 * RI);
    const uint32_t lt = (1u << lane) - 1u;

    uint32_t k[RI], pmv[RI];
#pragma unroll
    for (int i = 0; i < RI; ++i) {
        const uint32_t q = wbase + 32 * i + lane;
        k[i] = q < n ? skey[q] : 0u;
        pmv[i] = q < n ? sperm[q] : 0u;
    }
    // the row after the warp's last (lane 0 of the one after it too), the key
    // before the warp's first position and the key kPieceLen before it
    const uint32_t after = wbase + 32 * RI;
    const uint32_t halo = after + lane < n ? skey[after + lane] : 0u;
    const uint32_t halo2 = after + 32 < n ? skey[after + 32] : 0u;
    const uint32_t kprev = (wbase > 0 && wbase < n) ? skey[wbase - 1] : 0u;
    const uint32_t kback = (wbase >= 32 && wbase < n) ? skey[wbase - 32] : 0u;

    // position q is a segment head when it is 0 or its key differs from q-1's; a
    // piece head when it is a segment head, or a multiple of kPieceLen whose key
    // equals the key kPieceLen before it.  A head's segment spans several pieces
    // when the key at the first piece boundary at least kPieceLen past it (the
    // next row's lane 0 for lane 0, the row after for the others) is its own, and
    // is long when the key kShortLen past it is.
    uint32_t headm = 0, piecem = 0, multim = 0, longm = 0;
#pragma unroll
    for (int i = 0; i < RI; ++i) {
        const uint32_t q = wbase + 32 * i + lane;
        const uint32_t up = __shfl_up_sync(kFull, k[i], 1);
        const uint32_t row_before_last = (i == 0) ? kprev : __shfl_sync(kFull, k[i - 1], 31);
        const uint32_t back = (i == 0) ? kback : __shfl_sync(kFull, k[i - 1], 0);
        const uint32_t next_row = (i + 1 < RI) ? k[i + 1] : halo;
        const uint32_t next0 = __shfl_sync(kFull, next_row, 0);
        const uint32_t next1 = (i + 2 < RI) ? __shfl_sync(kFull, k[(i + 2) % RI], 0)
                                            : (i + 2 == RI ? __shfl_sync(kFull, halo, 0) : halo2);
        const uint32_t short_in = __shfl_down_sync(kFull, k[i], kShortLen);
        const uint32_t short_wrap = __shfl_sync(kFull, next_row, (lane + kShortLen) & 31);
        if (q < n) {
            const uint32_t before = lane ? up : row_before_last;
            const bool h = (q == 0) || (k[i] != before);
            const bool split = lane == 0 && q >= 32 && back == k[i];
            headm |= (h ? 1u : 0u) << i;
            piecem |= ((h || split) ? 1u : 0u) << i;
            if (h) {
                const uint32_t nxt = q - lane + (lane ? 64u : 32u);
                const bool multi = nxt < n && (lane ? next1 : next0) == k[i];
                const bool lng = q + kShortLen < n && (lane + kShortLen < 32 ? short_in : short_wrap) == k[i];
                multim |= (multi ? 1u : 0u) << i;
                longm |= (lng ? 1u : 0u) << i;
            }
        }
    }
    // last_step of each head's row (the step-order check), requested before the
    // scan and the look-back, whose round trips it overlaps
    int64_t last[RI];
#pragma unroll
    for (int i = 0; i < RI; ++i)
        last[i] = (((headm >> i) & 1u) && ls && !ls_per_coord && static_cast<int64_t>(k[i]) < bound) ? ls[k[i]] : 0;

    const uint32_t hcw = __reduce_add_sync(kFull, static_cast<unsigned>(__popc(headm)));
    const uint32_t pcw = __reduce_add_sync(kFull, static_cast<unsigned>(__popc(piecem)));
    if (lane == 0) s_warp[warp] = (hcw << 16) | pcw;
    __syncthreads();
    uint32_t wex = 0, tot = 0;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
        const uint32_t x = s_warp[w2];
        if (w2 < warp) wex += x;
        tot += x;
    }
    const unsigned long long agg = (static_cast<unsigned long long>(tot >> 16) << 31) | (tot & 0xffffu);

    if (tid < 32) {
        unsigned long long excl = 0;
        if (tile == 0) {
            if (lane == 0) st_volatile(dstatus + tile, (2ull << 62) | agg);
        } else {
            if (lane == 0) st_volatile(dstatus + tile, (1ull << 62) | agg);
            int64_t top = static_cast<int64_t>(tile) - 1;
            uint32_t spins = 0;
            while (true) {
                const int64_t jj = top - lane;
                unsigned long long w = (jj >= 0) ? ld_volatile(dstatus + jj) : (2ull << 62);
                while (__any_sync(kFull, (w >> 62) == 0ull)) {
                    if (++spins > kSpinLimit) {
                        if ((w >> 62) == 0ull) {
                            set_error(d_err, SPARSE_ERR_INTERNAL);
                            w = 2ull << 62;
                        }
                        continue;
                    }
                    if (spins > 64) __nanosleep(64);
                    if ((w >> 62) == 0ull) w = ld_volatile(dstatus + jj);
                }
                const uint32_t incl = __ballot_sync(kFull, (w >> 62) == 2ull);
                if (incl) {
                    const int first = __ffs(incl) - 1;
                    excl += warp_sum_u64(lane <= first ? (w & kValMask) : 0ull);
                    break;
                }
                excl += warp_sum_u64(w & kValMask);
                top -= 32;
            }
            if (lane == 0) st_volatile(dstatus + tile, (2ull << 62) | (excl + agg));
        }
        if (lane == 0) s_excl = excl;
    }
    __syncthreads();
    const unsigned long long ex = s_excl;
    uint32_t h_run = static_cast<uint32_t>(ex >> 31) + (wex >> 16);      // heads before the row
    uint32_t p_run = static_cast<uint32_t>(ex & 0x7fffffffull) + (wex & 0xffffu);

    uint32_t lists[RI];   // flagged pieces of this lane
    uint64_t kinds = 0;   // 3 bits per flagged piece: long, split head, group head
    int nl = 0;
#pragma unroll
    for (int i = 0; i < RI; ++i) {
        const uint32_t q = wbase + 32 * i + lane;
        const bool h = (headm >> i) & 1u;
        const bool ph = (piecem >> i) & 1u;
        const uint32_t hb = __ballot_sync(kFull, h);
        const uint32_t pb = __ballot_sync(kFull, ph);
        if (q < n) {
            const uint32_t u = h_run + __popc(hb & lt) + (h ? 1u : 0u) - 1u;  // segment of position q
            if (h) {
                seg_off[u] = q;
                if (idx_out) idx_out[u] = static_cast<int64_t>(k[i]);
                if (seg_off_out) seg_off_out[u] = static_cast<int64_t>(q);
                if (ls && static_cast<int64_t>(k[i]) < bound) {
                    if (!ls_per_coord) {
                        if (last[i] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
                    } else {
                        const int64_t b = static_cast<int64_t>(k[i]) * c;
                        for (int64_t jc = 0; jc < c; ++jc)
                            if (ls[b + jc] >= t) {
                                set_error(d_err, SPARSE_ERR_STEP_ORDER);
                                break;
                            }
                    }
                }
            }
            const uint32_t pm = pmv[i];
            if (perm_out) perm_out[q] = static_cast<int64_t>(pm);
            if (ph) {
                uint32_t flag = kMultiFlag;
                if (h) flag = ((multim >> i) & 1u) ? kMultiFlag : (((longm >> i) & 1u) ? kLongFlag : 0u);
                const uint32_t j = p_run + __popc(pb & lt);
                rec[j] = make_uint4(q, k[i], u | flag, pm);
                if (flag) {
                    lists[nl] = j;
                    kinds |= static_cast<uint64_t>((h && flag == kMultiFlag ? 2u : 0u) |
                                                   (flag == kMultiFlag && (h || q % (kPieceLen * kGroup) == 0) ? 4u : 0u) |
                                                   1u)
                             << (3 * nl);
                    ++nl;
                }
            }
        }
        h_run += __popc(hb);
        p_run += __popc(pb);
    }
    // the flagged pieces of the lane go to the long-piece, split-segment and
    // combine-group lists: one atomic per list and warp, the three in flight
    // together (lanes 0, 1, 2)
    uint32_t mine[3], incl[3], wtotal[3];
#pragma unroll
    for (int li = 0; li < 3; ++li) {
        mine[li] = 0;
        for (int e = 0; e < nl; ++e) mine[li] += static_cast<uint32_t>((kinds >> (3 * e + li)) & 1u);
        incl[li] = mine[li];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl[li], o);
            if (lane >= o) incl[li] += y;
        }
        wtotal[li] = __shfl_sync(kFull, incl[li], 31);
    }
    uint32_t basew = 0;
    if (lane < 3) {
        const uint32_t tot = lane == 0 ? wtotal[0] : lane == 1 ? wtotal[1] : wtotal[2];
        if (tot) basew = atomicAdd(counts + (lane == 0 ? kCntM : lane == 1 ? kCntS : kCntG), tot);
    }
#pragma unroll
    for (int li = 0; li < 3; ++li) {
        const uint32_t b = __shfl_sync(kFull, basew, li);
        uint32_t* dst = li == 0 ? mlist : li == 1 ? slist : glist;
        uint32_t at = b + incl[li] - mine[li];
        for (int e = 0; e < nl; ++e)
            if ((kinds >> (3 * e + li)) & 1u) dst[at++] = lists[e];
    }
    if (tile == gridDim.x - 1 && tid == 0) {
        const uint32_t U = static_cast<uint32_t>((ex + agg) >> 31);
        const uint32_t P = static_cast<uint32_t>((ex + agg) & 0x7fffffffull);
        counts[kCntU] = U;
        counts[kCntP] = P;
        seg_off[U] = n;
        rec[P] = make_uint4(n, 0u, 0u, 0u);
        if (seg_off_out) seg_off_out[U] = static_cast<int64_t>(n);
        if (d_nnz_out) *d_nnz_out = static_cast<int64_t>(U);
    }
}

cudaError_t sort_and_segment(const int64_t* idx, int64_t n, int64_t c, int64_t bound, const WsLayout& L,
                             SortWs& ws, int64_t* idx_out, int64_t* seg_off_out, int64_t* perm_out,
                             int64_t* d_nnz_out, const int64_t* ls, int ls_per_coord, int64_t t,
                             int32_t* d_err, cudaStream_t s)
{
    const uint32_t nn = static_cast<uint32_t>(n);
    {
        SO_PROFILE("range_hist", s);
        launch(k_range_hist, dim3(L.hist_blocks), dim3(kBlock), s, idx, nn, bound, L.passes, ws.bh,
               reinterpret_cast<uint4*>(ws.counts), static_cast<uint32_t>((L.ctrl_end - L.ctrl_begin) / 16),
               d_err);
    }
    for (int p = 0; p < L.passes; ++p) {
        const int out = p & 1;
        const int in = out ^ 1;
        uint32_t* st = ws.rstatus + static_cast<size_t>(p) * L.sort_tiles * 256;
        SO_PROFILE("radix_pass", s);
        const bool large = L.sort_items != kSortItems;
        const auto kern = p == 0 ? (large ? k_radix_pass<true, kSortItemsLarge> : k_radix_pass<true, kSortItems>)
                                 : (large ? k_radix_pass<false, kSortItemsLarge> : k_radix_pass<false, kSortItems>);
        if (p == 0)
            launch(kern, dim3(L.sort_tiles), dim3(kBlock), s, idx, nullptr, nullptr, ws.keys[out], ws.vals[out], nn,
                   8 * p, ws.bh, L.hist_blocks, ws.gh, L.passes, st, ws.counts + kCtrPass0 + p, d_err);
        else
            launch(kern, dim3(L.sort_tiles), dim3(kBlock), s, nullptr, ws.keys[in], ws.vals[in], ws.keys[out],
                   ws.vals[out], nn, 8 * p, ws.bh, L.hist_blocks, ws.gh + 256 * p, L.passes, st,
                   ws.counts + kCtrPass0 + p, d_err);
    }
    SO_PROFILE("run_detect", s);
    launch(L.run_items != kRunItems ? k_run_detect<kRunItemsLarge> : k_run_detect<kRunItems>, dim3(L.run_tiles),
           dim3(kBlock), s, ws.keys[ws.final_buf], ws.vals[ws.final_buf], nn, ws.rec,
                                                ws.seg_off, ws.mlist, ws.slist, ws.glist, ws.dstatus, ws.counts + kCtrRun, ws.counts,
                                                idx_out, seg_off_out, perm_out, d_nnz_out, ls, ls_per_coord,
                                                c, bound, t, d_err);
    return cudaGetLastError();
}

// Canonical row-COO check: rows strictly ascending in [0, r); last_step < t.
__global__ void __launch_bounds__(kBlock) k_check_rows(const int64_t* __restrict__ rows, int64_t n,
                                                       int64_t r, int64_t c, const int64_t* __restrict__ ls,
                                                       int ls_per_coord, int64_t t, int32_t* d_err)
{
    pdl_enter();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n; i += stride) {
        const int64_t k = rows[i];
        if (k < 0 || k >= r) {
            set_error(d_err, SPARSE_ERR_INDEX_OUT_OF_RANGE);
            continue;
        }
        if (i > 0 && rows[i - 1] >= k) set_error(d_err, SPARSE_ERR_NOT_CANONICAL);
        if (ls) {
            if (!ls_per_coord) {
                if (ls[k] >= t) set_error(d_err, SPARSE_ERR_STEP_ORDER);
            } else {
                for (int64_t j = 0; j < c; ++j)
                    if (ls[k * c + j] >= t) {
                        set_error(d_err, SPARSE_ERR_STEP_ORDER);
                        break;
                    }
            }
        }
    }
}

cudaError_t check_canonical_rows(const int64_t* rows, int64_t n, int64_t r, int64_t c, const int64_t* ls,
                                 int ls_per_coord, int64_t t, int32_t* d_err, cudaStream_t s)
{
    const int blocks = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>((n + kBlock - 1) / kBlock, 8 * num_sms())));
    SO_PROFILE("check_rows", s);
    launch(k_check_rows, dim3(blocks), dim3(kBlock), s, rows, n, r, c, ls, ls_per_coord, t, d_err);
    return cudaGetLastError();
}

}  // namespace so
