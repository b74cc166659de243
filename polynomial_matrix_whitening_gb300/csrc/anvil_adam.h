// anvil_adam.h -- parameter block of the Adam kernel (internal to libanvil).
#pragma once

#include <cuda_runtime.h>

namespace anvil {

struct AdamParams {
    float* p;
    const float* g;
    float* m;
    float* v;
    long long count;
    int vec;  // all four arrays 16-byte aligned: float4 path
    float beta1, beta2, c1, c2, eps, step_size, eff_wd;
};

cudaError_t launch_adam(const AdamParams& a, cudaStream_t stream);

}  // namespace anvil
