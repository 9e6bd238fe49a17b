// fused_sgd.cu -- lazy SGD (coupled weight decay, lazy momentum) row-fused
// launches.  "Module sparse_optimizer" (optirs-gpu 0.3.2 docs), "Sparse SGD".
#include "fused.cuh"

namespace so {

cudaError_t fused_rows_sgd_sorted(const SortWs& ws, const WsLayout& L, const float* vals, int64_t c,
                                  const SgdParams& P, int vec4, int32_t* d_err, cudaStream_t s)
{
    return launch_fused(sorted_src(ws), L.n, L.n > kPieceLen ? L.nb : 0, vals, c, SgdEpi{P, c}, ws.part, L.nb, vec4,
                        d_err, s);
}

cudaError_t fused_rows_sgd_canon(const int64_t* rows, int64_t n, const float* vals, int64_t c,
                                 const SgdParams& P, int vec4, int32_t* d_err, cudaStream_t s)
{
    return launch_fused(CanonSrc{rows, n}, n, 0, vals, c, SgdEpi{P, c}, nullptr, 0, vec4, d_err, s);
}

cudaError_t small_canon_sgd(const int64_t* rows, int64_t n, int64_t r, const float* vals, const SgdParams& P,
                            int32_t* d_err, cudaStream_t s)
{
    return launch_small_canon(rows, n, r, vals, SgdEpi{P, 1}, nullptr, 0, d_err, s);
}

}  // namespace so
