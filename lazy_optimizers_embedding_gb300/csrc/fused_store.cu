// fused_store.cu -- canonicalisation back half: the segmented sum of duplicate
// values written out as the canonical value rows.  "DiskSparseAdam (DSA)"
// README, "Safe Duplicate Aggregation & Sorted I/O".
#include "fused.cuh"

namespace so {

cudaError_t fused_rows_store_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                    const StoreParams& P, int vec4, int32_t* d_err, cudaStream_t s)
{
    return launch_fused(sorted_src(ws), L.n, L.n > kPieceLen ? L.nb : 0, vals, c, StoreEpi{P, c}, ws.part, L.nb, vec4,
                        d_err, s);
}

}  // namespace so
