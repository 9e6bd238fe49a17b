// static_ws.cu -- sparse_canonicalize_static_ws: the canonicalisation entry
// point for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace: code that runs inside
// a host application that owns every device allocation through its own pool,
// code built against a runtime where cudaMalloc is not permitted on the calling
// thread, or a plug-in that must not grow the process's memory footprint per
// call.  For them the scratch lives in one file-scope device array of fixed
// size, SPARSE_STATIC_WS_BYTES, that every GPU loading this library holds until
// the process exits.  The call allocates nothing.
//
// Host code cannot use the array's name as a device pointer (in host code it
// names a host-side shadow), so every call looks up the array's device address
// on the current device with cudaGetSymbolAddress.  The address is not cached:
// a cached one would go stale if the device's primary context were torn down
// and re-created (cudaDeviceReset), and the lookup is cheap once the module is
// loaded.  Under lazy module loading the first lookup on a device is what loads
// the library's device code there, and with it creates the array.
#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[SPARSE_STATIC_WS_BYTES];

}  // namespace

extern "C" sparse_status_t sparse_canonicalize_static_ws(const int64_t* idx, const float* vals, int64_t n,
                                                         int64_t c, int64_t bound, int64_t* idx_out,
                                                         float* vals_out, int64_t* seg_off_out, int64_t* perm_out,
                                                         int64_t* d_nnz_out, int32_t* d_err, cudaStream_t stream)
{
    if (n < 0 || c < 1 || bound < 1) return SPARSE_ERR_INVALID_ARG;
    if (sparse_workspace_size(n, c, bound) > static_cast<size_t>(SPARSE_STATIC_WS_BYTES))
        return SPARSE_ERR_WORKSPACE;
    void* ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_static_ws) != cudaSuccess || ws == nullptr) return SPARSE_ERR_CUDA;
    return sparse_canonicalize(idx, vals, n, c, bound, idx_out, vals_out, seg_off_out, perm_out, d_nnz_out, ws,
                               static_cast<size_t>(SPARSE_STATIC_WS_BYTES), d_err, stream);
}
