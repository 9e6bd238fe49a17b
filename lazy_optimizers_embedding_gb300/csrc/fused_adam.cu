// fused_adam.cu -- lazy Adam (Lazy and DormancyDecay) row-fused launches:
// raw input (sorted segments, duplicates summed in the same pass) and
// canonical row-COO.  "Module sparse_optimizer" (optirs-gpu 0.3.2 docs), "Lazy Adam".
#include "fused.cuh"

namespace so {

cudaError_t fused_rows_adam_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                   const AdamParams& P, int vec4, int32_t* d_err, cudaStream_t s)
{
    return launch_fused(sorted_src(ws), L.n, L.n > kPieceLen ? L.nb : 0, vals, c, AdamEpi{P, c}, ws.part, L.nb,
                        vec4, d_err, s);
}

cudaError_t fused_rows_adam_canon(const int64_t* rows, int64_t n, const float* vals, int64_t c,
                                  const AdamParams& P, int vec4, int32_t* d_err, cudaStream_t s)
{
    return launch_fused(CanonSrc{rows, n}, n, 0, vals, c, AdamEpi{P, c}, nullptr, 0, vec4, d_err, s);
}

}  // namespace so
