// profile.cuh -- launch-site hook of the optional per-kernel timing.
#pragma once

#include <cuda_runtime.h>

namespace so {
namespace prof {

bool enabled();

// Records a start event on construction and a stop event on destruction, on the
// given stream, when profiling is enabled; does nothing otherwise.
class Scope {
public:
    Scope(const char* name, cudaStream_t s);
    ~Scope();
    Scope(const Scope&) = delete;
    Scope& operator=(const Scope&) = delete;

private:
    const char* name_;
    cudaStream_t stream_;
    cudaEvent_t start_;
};

}  // namespace prof
}  // namespace so

#define SO_PROFILE(name, stream) ::so::prof::Scope so_profile_scope_(name, stream)
