// anvil_adam.cu -- the Adam step with cautious weight decay that the page uses for the
// parameters outside the ANVIL banks (page "modded-nanogpt track_1_short/optim/anvil.py",
// `_adam_update_step`), as one HBM-bound elementwise kernel: 16 bytes read and 12 bytes
// written per element, four elements per thread per iteration (one 16-byte vector of
// each array).  Every rounding follows the page's fp32 tensor operations one at a time.
#include <cuda_runtime.h>
#include <stdint.h>

#include "anvil_adam.h"

namespace anvil {

__device__ __forceinline__ void adam_element(float& p, float g, float& m, float& v, const AdamParams& a) {
    m = __fadd_rn(__fmul_rn(m, a.beta1), __fmul_rn(a.c1, g));
    v = __fadd_rn(__fmul_rn(v, a.beta2), __fmul_rn(__fmul_rn(a.c2, g), g));
    float u = __fmul_rn(__fdiv_rn(m, __fadd_rn(__fsqrt_rn(v), a.eps)), a.step_size);
    const float mask = (__fmul_rn(u, p) > 0.f) ? 1.f : 0.f;
    u = __fadd_rn(u, __fmul_rn(__fmul_rn(a.eff_wd, p), mask));
    p = __fsub_rn(p, u);
}

__global__ void __launch_bounds__(256) adam_kernel(const AdamParams a) {
    const long long nvec = a.vec ? a.count / 4 : 0;  // float4 vectors (aligned path)
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nvec; i += stride) {
        float4 p = reinterpret_cast<float4*>(a.p)[i];
        const float4 g = __ldcs(reinterpret_cast<const float4*>(a.g) + i);
        float4 m = reinterpret_cast<float4*>(a.m)[i];
        float4 v = reinterpret_cast<float4*>(a.v)[i];
        adam_element(p.x, g.x, m.x, v.x, a);
        adam_element(p.y, g.y, m.y, v.y, a);
        adam_element(p.z, g.z, m.z, v.z, a);
        adam_element(p.w, g.w, m.w, v.w, a);
        reinterpret_cast<float4*>(a.p)[i] = p;
        reinterpret_cast<float4*>(a.m)[i] = m;
        reinterpret_cast<float4*>(a.v)[i] = v;
    }
    // the tail that is not a whole vector (or everything when unaligned)
    for (long long e = 4 * nvec + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < a.count;
         e += stride) {
        float p = a.p[e], m = a.m[e], v = a.v[e];
        adam_element(p, a.g[e], m, v, a);
        a.p[e] = p;
        a.m[e] = m;
        a.v[e] = v;
    }
}

cudaError_t launch_adam(const AdamParams& a, cudaStream_t stream) {
    // grid-stride, at most 16 blocks for each of a GB300's 152 SMs: 2.67 waves of the
    // resident blocks, measured faster than one, two or three whole waves
    long long blocks = (a.count / 4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    adam_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace anvil
