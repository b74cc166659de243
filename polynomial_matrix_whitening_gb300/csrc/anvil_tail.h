// anvil_tail.h -- parameter blocks of the update-tail kernels (internal to libanvil).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace anvil {

struct TailBank {
    const uint16_t* update;   // [g, m, n] bf16: the cascade output
    const float* velocity;    // [2, g, m, n]: rail 1 (slow) gates the decay
    float* lane_energy;       // [g, nl] fp32 state, nl = m if m >= n else n
    uint16_t* param;          // [g, m, n] bf16 bits of the master weight (high half)
    uint16_t* mantissa;       // [g, m, n] low half of the master weight
    const float* eff_lr;      // [g] per-matrix learning rate (device)
    float eff_wd, beta2;
    int g, m, n;
    int mat_begin;            // first matrix of this bank in the call
    long long chunk_begin;    // first 8-element row chunk of this bank in the call
    long long row_begin;      // first row of this bank in the call (g * m rows per bank)
    long long power_begin;    // first block of this bank in the lane-power grid (set by its launcher)
    int power_nblk;           // lanes along rows: blocks of this bank in the lane-power grid (set by its launcher)
    int vec8;                 // n % 8 == 0 and 16-byte aligned buffers: vector path
    float* power;             // workspace [g, nl]: lane powers
    float* scale;             // workspace [g, nl]: bf16-rounded lane scales
    const uint64_t* sign;     // tail link slow-rail sign words [g, nck, m, 2] (NULL: read the rail)
    int nck;
};

struct TailParams {
    TailBank bank[8];
    int nbanks, total_mats;
    long long total_chunks, total_rows;
};

cudaError_t launch_tail_power(const TailParams& p, cudaStream_t stream);
cudaError_t launch_tail_scale(const TailParams& p, cudaStream_t stream);
cudaError_t launch_tail_apply(const TailParams& p, cudaStream_t stream);

}  // namespace anvil
