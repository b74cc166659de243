// anvil_tail.cu -- the update tail after the cascade (page "modded-nanogpt
// track_1_short/optim/anvil.py", `anvil_bank_update` steps 2 and 3: `_rail_equalizer` and
// `_sign_aligned_decay_update`), three HBM-bound kernels grouped over banks:
//
//   lane_power_kernel : P[l] = mean over lane l of float(v)^2; lanes run along the longer
//                       dimension (rows when m >= n, else columns)
//   lane_scale_kernel : one block per matrix: lane_energy <- lerp(lane_energy, P, 1 - beta2),
//                       gain = rsqrt(max(lane_energy, 1e-10)), norms before and after,
//                       scale[l] = bf16(gain * (pre_norm / max(post_norm, 1e-10)))
//   tail_apply_kernel : u = bf16(v * scale[lane]); on the fp32 master weight w (bf16 bits
//                       p, uint16 mantissa): w <- (w - w [gate w >= 0] wd lr) - u lr, split
//                       back into p and mantissa (gate: the slow rail)
//   tail_apply_rows_kernel : the same, the gate taken from the sign bits that the step
//                       left in the tail link (the fp32 rail only where they cannot decide)
//
// Every rounding follows the page's fp32 tensor operations one at a time (no FMA; the
// linked apply takes two elements per packed fp32 operation, two such roundings).
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/anvil.h"
#include "anvil_device.cuh"
#include "anvil_internal.h"
#include "anvil_tail.h"

namespace anvil {

// ---------------------------------------------------------------- lane powers
// One grid over every bank (a block finds its bank from power_begin).
// Lanes along rows (m >= n): a warp sums groups of POWER_ROWS consecutive rows of the bank
// (rows of consecutive matrices are contiguous), the bank's power_nblk blocks walking its
// groups with a stride of their warps; with the vector layout (n % 8 == 0, 16-byte
// aligned) lane k takes 8-element chunks k, k + 32, ... of every row, POWER_CHUNKS chunks
// of each of the group's rows loaded before any is summed (one memory round trip for rows
// of up to 768 elements, and then the next group's loads go out before this group's sums
// are reduced), otherwise single elements; a fixed shuffle tree adds each row's 32
// partial sums.
// Lanes along columns (m < n): a block covers 256 columns of one matrix (8 per thread with
// the vector layout, else 32 columns) with 8 row slices; slice k sums rows k, k + 8, ...;
// the slice sums of a column are added in slice order.
constexpr int POWER_COLS = 256;  // columns per block, lanes along columns, vector layout
constexpr int POWER_ROWS = 2;    // rows per group, lanes along rows
constexpr int POWER_CHUNKS = 3;  // 16-byte chunks of each row a lane loads before summing
__device__ __forceinline__ float sumsq8(uint4 q, float s) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float x = bf2f(static_cast<uint16_t>((k & 1) ? w[k >> 1] >> 16 : w[k >> 1] & 0xffffu));
        s = __fadd_rn(s, __fmul_rn(x, x));
    }
    return s;
}
__host__ __device__ inline long long power_groups(const TailBank& B) {
    return (static_cast<long long>(B.g) * B.m + POWER_ROWS - 1) / POWER_ROWS;
}
__host__ __device__ inline long long power_blocks(const TailBank& B) {
    if (B.m >= B.n) return B.power_nblk;
    const int span = B.vec8 ? POWER_COLS : 32;
    return static_cast<long long>(B.g) * ((B.n + span - 1) / span);
}
__global__ void __launch_bounds__(256, 4) lane_power_kernel(const __grid_constant__ TailParams p) {
    pdl_allow_next();
    pdl_wait_previous();
    const long long blk = blockIdx.x;
    int b = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (blk >= p.bank[i].power_begin) b = i;
    const TailBank& B = p.bank[b];
    const long long lb = blk - B.power_begin;
    if (B.m >= B.n) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const long long nrows = static_cast<long long>(B.g) * B.m;
        const long long ngroups = power_groups(B), gstride = static_cast<long long>(B.power_nblk) * 8;
        long long grp = lb * 8 + warp;
        if (grp >= ngroups) return;  // whole warp
        const int nc = B.n / 8;
        // the group's row sums, reduced across the warp and stored (lane 0)
        auto finish = [&](long long row0, float (&s)[POWER_ROWS]) {
#pragma unroll
            for (int k = 0; k < POWER_ROWS; ++k) {
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1) s[k] = __fadd_rn(s[k], __shfl_xor_sync(0xffffffffu, s[k], off));
                if (lane == 0 && row0 + k < nrows) B.power[row0 + k] = __fdiv_rn(s[k], static_cast<float>(B.n));
            }
        };
        if (B.vec8 && nc <= 32 * POWER_CHUNKS) {
            // one load round per group: group grp + gstride's loads go out before grp's reduction
            uint4 q[POWER_CHUNKS][POWER_ROWS];
            auto load = [&](long long row0) {
#pragma unroll
                for (int u = 0; u < POWER_CHUNKS; ++u)
#pragma unroll
                    for (int k = 0; k < POWER_ROWS; ++k)
                        q[u][k] = (lane + 32 * u < nc && row0 + k < nrows)
                                      ? __ldcs(reinterpret_cast<const uint4*>(B.update + static_cast<size_t>(row0 + k) * B.n) + lane + 32 * u)
                                      : make_uint4(0u, 0u, 0u, 0u);
            };
            load(grp * POWER_ROWS);
            for (;;) {
                float s[POWER_ROWS];
#pragma unroll
                for (int k = 0; k < POWER_ROWS; ++k) s[k] = 0.f;
#pragma unroll
                for (int u = 0; u < POWER_CHUNKS; ++u)
#pragma unroll
                    for (int k = 0; k < POWER_ROWS; ++k) s[k] = sumsq8(q[u][k], s[k]);
                const long long nxt = grp + gstride;
                if (nxt < ngroups) load(nxt * POWER_ROWS);
                finish(grp * POWER_ROWS, s);
                if (nxt >= ngroups) break;
                grp = nxt;
            }
            return;
        }
        for (; grp < ngroups; grp += gstride) {
        const long long row0 = grp * POWER_ROWS;  // row (mat * m + row) of the bank
        float s[POWER_ROWS];
#pragma unroll
        for (int k = 0; k < POWER_ROWS; ++k) s[k] = 0.f;
        if (B.vec8) {
            for (int j0 = lane; j0 < nc; j0 += 32 * POWER_CHUNKS) {
                uint4 q[POWER_CHUNKS][POWER_ROWS];
#pragma unroll
                for (int u = 0; u < POWER_CHUNKS; ++u)
#pragma unroll
                    for (int k = 0; k < POWER_ROWS; ++k)
                        q[u][k] = (j0 + 32 * u < nc && row0 + k < nrows)
                                      ? __ldcs(reinterpret_cast<const uint4*>(B.update + static_cast<size_t>(row0 + k) * B.n) + j0 + 32 * u)
                                      : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < POWER_CHUNKS; ++u)
#pragma unroll
                    for (int k = 0; k < POWER_ROWS; ++k) s[k] = sumsq8(q[u][k], s[k]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < POWER_ROWS; ++k) {
                if (row0 + k >= nrows) break;
                const uint16_t* v = B.update + static_cast<size_t>(row0 + k) * B.n;
                for (int j = lane; j < B.n; j += 32) {
                    const float x = bf2f(v[j]);
                    s[k] = __fadd_rn(s[k], __fmul_rn(x, x));
                }
            }
        }
        finish(row0, s);
        }
    } else {
        __shared__ float part[8][POWER_COLS + 1];
        const int span = B.vec8 ? POWER_COLS : 32;  // columns per block
        const int cblocks = (B.n + span - 1) / span;
        const int mat = static_cast<int>(lb / cblocks), c0 = static_cast<int>(lb % cblocks) * span;
        const int cx = threadIdx.x & 31, slice = threadIdx.x >> 5;
        const uint16_t* v = B.update + static_cast<size_t>(mat) * B.m * B.n;
        if (B.vec8) {
            // thread: columns c0 + 8 cx .. +7 (n % 8 == 0, so a chunk is in or out whole)
            const int col = c0 + 8 * cx;
            float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (col < B.n)
                // rows slice, slice + 8, ... in that order, eight rows' loads in flight at once
                for (int i0 = slice; i0 < B.m; i0 += 64) {
                    uint4 q[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int i = i0 + 8 * u;
                        q[u] = i < B.m ? __ldcs(reinterpret_cast<const uint4*>(v + static_cast<size_t>(i) * B.n + col))
                                       : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (i0 + 8 * u >= B.m) break;
                        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float x = bf2f(static_cast<uint16_t>((k & 1) ? w[k >> 1] >> 16 : w[k >> 1] & 0xffffu));
                            s[k] = __fadd_rn(s[k], __fmul_rn(x, x));
                        }
                    }
                }
#pragma unroll
            for (int k = 0; k < 8; ++k) part[slice][8 * cx + k] = s[k];
            __syncthreads();
            const int c = c0 + threadIdx.x;  // one column per thread
            if (c < B.n) {
                float t = part[0][threadIdx.x];
                for (int k = 1; k < 8; ++k) t = __fadd_rn(t, part[k][threadIdx.x]);
                B.power[static_cast<size_t>(mat) * B.n + c] = __fdiv_rn(t, static_cast<float>(B.m));
            }
        } else {
            const int col = c0 + cx;
            float s = 0.f;
            if (col < B.n)
                for (int i = slice; i < B.m; i += 8) {
                    const float x = bf2f(v[static_cast<size_t>(i) * B.n + col]);
                    s = __fadd_rn(s, __fmul_rn(x, x));
                }
            part[slice][cx] = s;
            __syncthreads();
            if (slice == 0 && col < B.n) {
                float t = part[0][cx];
                for (int k = 1; k < 8; ++k) t = __fadd_rn(t, part[k][cx]);
                B.power[static_cast<size_t>(mat) * B.n + col] = __fdiv_rn(t, static_cast<float>(B.m));
            }
        }
    }
}

// ---------------------------------------------------------------- lane scales
// One block per matrix; sums in a fixed order (per thread, per warp by shuffles, then
// over the warps).
constexpr int SCALE_THREADS = 1024;
__global__ void __launch_bounds__(SCALE_THREADS) lane_scale_kernel(const __grid_constant__ TailParams p) {
    __shared__ float red_p[SCALE_THREADS / 32], red_q[SCALE_THREADS / 32];
    __shared__ float ratio_s;
    pdl_allow_next();
    pdl_wait_previous();
    const int gm = blockIdx.x;
    int bi = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (gm >= p.bank[i].mat_begin) bi = i;
    const TailBank& B = p.bank[bi];
    const int mat = gm - B.mat_begin;
    const int nl = B.m >= B.n ? B.m : B.n;
    const float len = static_cast<float>(B.m >= B.n ? B.n : B.m);
    const float w = __fsub_rn(1.0f, B.beta2);
    const float* P = B.power + static_cast<size_t>(mat) * nl;
    float* E = B.lane_energy + static_cast<size_t>(mat) * nl;
    float* S = B.scale + static_cast<size_t>(mat) * nl;
    float sp = 0.f, sq = 0.f;
    for (int l = threadIdx.x; l < nl; l += SCALE_THREADS) {
        const float pw = P[l];
        const float e0 = E[l];
        const float e = __fadd_rn(e0, __fmul_rn(w, __fsub_rn(pw, e0)));
        E[l] = e;
        const float gain = __frsqrt_rn(e > 1e-10f ? e : 1e-10f);
        S[l] = gain;
        sp = __fadd_rn(sp, pw);
        sq = __fadd_rn(sq, __fmul_rn(__fmul_rn(pw, len), __fmul_rn(gain, gain)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sp = __fadd_rn(sp, __shfl_xor_sync(0xffffffffu, sp, o));
        sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, o));
    }
    if ((threadIdx.x & 31) == 0) {
        red_p[threadIdx.x >> 5] = sp;
        red_q[threadIdx.x >> 5] = sq;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        float a = red_p[threadIdx.x], c = red_q[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
            c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, o));
        }
        if (threadIdx.x == 0) {
            const float pre = __fsqrt_rn(__fmul_rn(a, len));
            float post = __fsqrt_rn(c);
            if (post < 1e-10f) post = 1e-10f;
            ratio_s = __fdiv_rn(pre, post);
        }
    }
    __syncthreads();
    const float ratio = ratio_s;
    for (int l = threadIdx.x; l < nl; l += SCALE_THREADS) S[l] = round_bf(__fmul_rn(S[l], ratio));
}

// ---------------------------------------------------------------- equalise + decay update
__device__ __forceinline__ void tail_element(float v, float scale, float gate, float wd, float lr,
                                             uint16_t& p, uint16_t& mt) {
    const float u = round_bf(__fmul_rn(v, scale));
    float w = __uint_as_float((static_cast<uint32_t>(p) << 16) | mt);
    const float aligned = (__fmul_rn(gate, w) >= 0.f) ? 1.f : 0.f;
    const float decay = __fmul_rn(__fmul_rn(__fmul_rn(w, aligned), wd), lr);
    w = __fsub_rn(__fsub_rn(w, decay), __fmul_rn(u, lr));
    const uint32_t bits = __float_as_uint(w);
    p = static_cast<uint16_t>(bits >> 16);
    mt = static_cast<uint16_t>(bits & 0xffffu);
}

// Eight consecutive elements of one row per thread, grid-stride over all banks.
__global__ void __launch_bounds__(256) tail_apply_kernel(const __grid_constant__ TailParams p) {
    pdl_allow_next();
    pdl_wait_previous();
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < p.total_chunks;
         t += stride) {
        int bi = 0;
#pragma unroll 1
        for (int i = 1; i < p.nbanks; ++i)
            if (t >= p.bank[i].chunk_begin) bi = i;
        const TailBank& B = p.bank[bi];
        const long long lt = t - B.chunk_begin;
        const int cpr = (B.n + 7) / 8;  // chunks per row
        int mat, row, c0;
        if (lt < 0x7fffffffLL) {
            // 32-bit division (the common case: a bank of under 2^31 chunks)
            const unsigned l = static_cast<unsigned>(lt), ucpr = static_cast<unsigned>(cpr);
            const unsigned rowg = l / ucpr;
            c0 = static_cast<int>(l - rowg * ucpr) * 8;
            mat = static_cast<int>(rowg / static_cast<unsigned>(B.m));
            row = static_cast<int>(rowg - static_cast<unsigned>(mat) * static_cast<unsigned>(B.m));
        } else {
            const long long rowg = lt / cpr;
            c0 = static_cast<int>(lt % cpr) * 8;
            mat = static_cast<int>(rowg / B.m);
            row = static_cast<int>(rowg % B.m);
        }
        const size_t mn = static_cast<size_t>(B.m) * B.n;
        const size_t base = static_cast<size_t>(mat) * mn + static_cast<size_t>(row) * B.n + c0;
        const float lr = B.eff_lr[mat];
        const bool rows_lanes = B.m >= B.n;
        const float* S = B.scale + static_cast<size_t>(mat) * (rows_lanes ? B.m : B.n);
        const float* gate = B.velocity + static_cast<size_t>(B.g) * mn;  // rail 1
        if (B.vec8 && c0 + 8 <= B.n) {
            const uint4 vu = *reinterpret_cast<const uint4*>(B.update + base);
            uint4 pu = *reinterpret_cast<const uint4*>(B.param + base);
            uint4 mu = *reinterpret_cast<const uint4*>(B.mantissa + base);
            const float4 g0 = __ldcs(reinterpret_cast<const float4*>(gate + base));
            const float4 g1 = __ldcs(reinterpret_cast<const float4*>(gate + base + 4));
            const uint32_t vw[4] = {vu.x, vu.y, vu.z, vu.w};
            uint32_t pw[4] = {pu.x, pu.y, pu.z, pu.w};
            uint32_t mw[4] = {mu.x, mu.y, mu.z, mu.w};
            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int q = k >> 1, hi = k & 1;
                const float v = bf2f(static_cast<uint16_t>(hi ? vw[q] >> 16 : vw[q] & 0xffffu));
                uint16_t pp = static_cast<uint16_t>(hi ? pw[q] >> 16 : pw[q] & 0xffffu);
                uint16_t mm = static_cast<uint16_t>(hi ? mw[q] >> 16 : mw[q] & 0xffffu);
                tail_element(v, rows_lanes ? S[row] : S[c0 + k], gv[k], B.eff_wd, lr, pp, mm);
                pw[q] = hi ? ((pw[q] & 0xffffu) | (static_cast<uint32_t>(pp) << 16))
                           : ((pw[q] & 0xffff0000u) | pp);
                mw[q] = hi ? ((mw[q] & 0xffffu) | (static_cast<uint32_t>(mm) << 16))
                           : ((mw[q] & 0xffff0000u) | mm);
            }
            *reinterpret_cast<uint4*>(B.param + base) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
            *reinterpret_cast<uint4*>(B.mantissa + base) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
        } else {
            for (int k = 0; k < 8 && c0 + k < B.n; ++k) {
                uint16_t pp = B.param[base + k], mm = B.mantissa[base + k];
                tail_element(bf2f(B.update[base + k]), rows_lanes ? S[row] : S[c0 + k], gate[base + k],
                             B.eff_wd, lr, pp, mm);
                B.param[base + k] = pp;
                B.mantissa[base + k] = mm;
            }
        }
    }
}

// tail_element with the gate already decided (the tail link's path).
__device__ __forceinline__ void tail_element_gated(float v, float scale, bool aligned_, float wd, float lr,
                                                   uint16_t& p, uint16_t& mt) {
    const float u = round_bf(__fmul_rn(v, scale));
    float w = __uint_as_float((static_cast<uint32_t>(p) << 16) | mt);
    const float aligned = aligned_ ? 1.f : 0.f;
    const float decay = __fmul_rn(__fmul_rn(__fmul_rn(w, aligned), wd), lr);
    w = __fsub_rn(__fsub_rn(w, decay), __fmul_rn(u, lr));
    const uint32_t bits = __float_as_uint(w);
    p = static_cast<uint16_t>(bits >> 16);
    mt = static_cast<uint16_t>(bits & 0xffffu);
}

// The 8 bits of columns 4 t .. 4 t + 7 of a link word (bit 16 q + t is column 4 t + q), in
// column order: the bits at 0, 16, 32, 48 of (w >> t) gathered by one multiply.
__device__ __forceinline__ unsigned link_bits8(uint64_t w, int t) {
    const uint64_t lo = (w >> t) & 0x0001000100010001ull, hi = (w >> (t + 1)) & 0x0001000100010001ull;
    constexpr uint64_t M = (1ull << 48) | (1ull << 33) | (1ull << 18) | (1ull << 3);
    return static_cast<unsigned>(((lo * M) >> 48) & 0xfu) | (static_cast<unsigned>(((hi * M) >> 48) & 0xfu) << 4);
}


// The gate bits of a chunk, in the order the link words give them up cheaply: element k
// of the chunk at bit gate_pos(k).  Before the last fold the bits sit "spread" at bit
// 16 (k & 1) + 2 ((k >> 1) & 1) + (k >> 2) of a word, which gathers them from a link word
// (bit 16 q + t of the word is column 4 t + q of its 64 columns) with two 32-bit shifts.
__host__ __device__ constexpr int gate_pos(int k) { return 4 * (k & 1) + 2 * ((k >> 1) & 1) + (k >> 2); }
// The spread bits of chunk j (columns 8 j .. 8 j + 7) of a link word.
__device__ __forceinline__ uint32_t link_spread(uint64_t w, int j) {
    const uint32_t a = static_cast<uint32_t>(w) >> (2 * j), b = static_cast<uint32_t>(w >> 32) >> (2 * j);
    return (a & 0x00030003u) | ((b & 0x00030003u) << 2);
}
// The spread sign bits of the chunk's master weights (bit 15 and 31 of each param word
// are the signs of elements 2 q and 2 q + 1).
__device__ __forceinline__ uint32_t sign_spread(const uint32_t (&pw)[4]) {
    return ((pw[0] >> 15) & 0x00010001u) | ((pw[2] >> 14) & 0x00020002u) | ((pw[1] >> 13) & 0x00040004u) |
           ((pw[3] >> 12) & 0x00080008u);
}
__device__ __forceinline__ unsigned fold_spread(uint32_t x) { return (x | (x >> 12)) & 0xffu; }

// With the tail link: the decay gate [slow rail * w >= 0] of an element follows from the
// sign bits (the product of two numbers of magnitude at least 2^-100 and 2^-40 is not zero
// and has the sign of their signs) unless the link flags the rail value (zero, below
// 2^-100, not finite) or w is outside [2^-40, FLT_MAX] (its exponent field outside
// [87, 254]): then the fp32 rail is read.  Result: element k aligned at bit gate_pos(k).
__device__ __forceinline__ unsigned link_gates(ulonglong2 sx, int c0, const float* rail, const uint32_t (&pw)[4],
                                               const uint32_t (&mw)[4]) {
    const int j = (c0 & 63) >> 3;  // the chunk's 8 of the link word's 64 columns
    const uint32_t g = link_spread(sx.x, j);
    bool need_rail = link_spread(sx.y, j) != 0u;
    // exponent fields e of both halves of every param word: e + 169 reaches bit 8 iff
    // e >= 87, e + 1 iff e = 255 (no carry crosses into the upper half)
    uint32_t ge87 = 0xffffffffu, is255 = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t e2 = (pw[q] >> 7) & 0x00ff00ffu;
        ge87 &= e2 + 0x00a900a9u;
        is255 |= e2 + 0x00010001u;
    }
    need_rail |= ((~ge87 | is255) & 0x01000100u) != 0u;
    if (!need_rail) return fold_spread(~(g ^ sign_spread(pw)) & 0x000f000fu);
    const float4 r0 = __ldcs(reinterpret_cast<const float4*>(rail));
    const float4 r1 = __ldcs(reinterpret_cast<const float4*>(rail + 4));
    const float rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    unsigned gk = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int q = k >> 1, hi = k & 1;
        const float w = __uint_as_float((hi ? (pw[q] & 0xffff0000u) : (pw[q] << 16)) | (hi ? (mw[q] >> 16) : (mw[q] & 0xffffu)));
        gk |= (__fmul_rn(rv[k], w) >= 0.f ? 1u : 0u) << gate_pos(k);
    }
    return gk;
}

// Lane scales of a chunk as pairs: the row's scale sr (lanes along rows), else the
// chunk's 8 column scales at S (16-byte aligned).
__device__ __forceinline__ void scale_pairs(uint64_t (&sc2)[4], bool rows_lanes, float sr, const float* S) {
    if (rows_lanes) {
        const uint64_t r2 = f2_pack(sr, sr);
#pragma unroll
        for (int q = 0; q < 4; ++q) sc2[q] = r2;
    } else {
        const float4 s0 = *reinterpret_cast<const float4*>(S);
        const float4 s1 = *reinterpret_cast<const float4*>(S + 4);
        sc2[0] = f2_pack(s0.x, s0.y);
        sc2[1] = f2_pack(s0.z, s0.w);
        sc2[2] = f2_pack(s1.x, s1.y);
        sc2[3] = f2_pack(s1.z, s1.w);
    }
}

// Eight elements of one row chunk (bf16 update words vw, master-weight words pw and mw,
// lane-scale pairs sc2, gate bits gk at gate_pos), updated in place, two elements per
// packed fp32 operation (each half an IEEE round-to-nearest operation, in the order of
// tail_element_gated): u = bf16(v s); w <- (w - w [gate] wd lr) - u lr.
__device__ __forceinline__ void apply8_gated(const uint32_t (&vw)[4], uint32_t (&pw)[4], uint32_t (&mw)[4],
                                             const uint64_t (&sc2)[4], unsigned gk, float wd, float lr) {
    const uint64_t wd2 = f2_pack(wd, wd), lr2 = f2_pack(lr, lr);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint64_t u2 = bf2_to_f2(f2_to_bf2(f2_mul(bf2_to_f2(vw[q]), sc2[q])));
        // w of elements 2 q and 2 q + 1: param bits above, mantissa below
        const uint32_t w0 = __byte_perm(mw[q], pw[q], 0x5410), w1 = __byte_perm(mw[q], pw[q], 0x7632);
        const uint64_t w2 = (static_cast<uint64_t>(w1) << 32) | w0;
        const uint64_t al2 = f2_pack((gk >> gate_pos(2 * q)) & 1u ? 1.f : 0.f, (gk >> gate_pos(2 * q + 1)) & 1u ? 1.f : 0.f);
        const uint64_t decay = f2_mul(f2_mul(f2_mul(w2, al2), wd2), lr2);
        const uint64_t r = f2_add(f2_add(w2, f2_neg(decay)), f2_neg(f2_mul(u2, lr2)));
        const uint32_t r0 = static_cast<uint32_t>(r), r1 = static_cast<uint32_t>(r >> 32);
        pw[q] = __byte_perm(r0, r1, 0x7632);
        mw[q] = __byte_perm(r0, r1, 0x5410);
    }
}

// With every bank's link: one warp per row at a time (grid-stride over the call's rows),
// lane l taking the 8-element chunks l, l + 32, ... of the row, ROW_CHUNKS of them loaded
// before any is computed (one: more chunks per lane need more registers than five blocks
// per SM leave, and spilled or cost occupancy; both measured slower).  The row's matrix,
// learning rate and (rows as lanes) scale are found once per row.
constexpr int ROW_CHUNKS = 1;
__global__ void __launch_bounds__(256, 5) tail_apply_rows_kernel(const __grid_constant__ TailParams p) {
    pdl_allow_next();
    pdl_wait_previous();
    const int lane = threadIdx.x & 31;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    for (long long rw = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); rw < p.total_rows;
         rw += nwarps) {
        int bi = 0;
#pragma unroll 1
        for (int i = 1; i < p.nbanks; ++i)
            if (rw >= p.bank[i].row_begin) bi = i;
        const TailBank& B = p.bank[bi];
        // a bank has at most ANVIL_MAX_BATCH * ANVIL_MAX_DIM < 2^31 rows: 32-bit division
        const unsigned lrow = static_cast<unsigned>(rw - B.row_begin);
        const int mat = static_cast<int>(lrow / static_cast<unsigned>(B.m));
        const int row = static_cast<int>(lrow - static_cast<unsigned>(mat) * static_cast<unsigned>(B.m));
        const size_t rbase = (static_cast<size_t>(mat) * B.m + row) * B.n;
        const float lr = B.eff_lr[mat];
        const bool rows_lanes = B.m >= B.n;
        const float* S = B.scale + static_cast<size_t>(mat) * (rows_lanes ? B.m : B.n);
        const float srow = rows_lanes ? S[row] : 0.f;
        const float* rail = B.velocity + static_cast<size_t>(B.g) * B.m * B.n + rbase;
        // the row's sign words of 64-column chunk k: sgn + 2 m k ([g, nck, m, 2])
        const uint64_t* sgn = B.sign + (static_cast<size_t>(mat) * B.nck * B.m + row) * 2;
        const size_t kstride = 2 * static_cast<size_t>(B.m);
        const int nch = (B.n + 7) / 8;
        for (int cb = lane; cb < nch; cb += 32 * ROW_CHUNKS) {
            uint4 vu[ROW_CHUNKS], pu[ROW_CHUNKS], mu[ROW_CHUNKS];
            ulonglong2 sx[ROW_CHUNKS];
#pragma unroll
            for (int u = 0; u < ROW_CHUNKS; ++u) {
                const int ci = cb + 32 * u;
                if (B.vec8 && ci < nch) {
                    vu[u] = *reinterpret_cast<const uint4*>(B.update + rbase + 8 * ci);
                    pu[u] = *reinterpret_cast<const uint4*>(B.param + rbase + 8 * ci);
                    mu[u] = *reinterpret_cast<const uint4*>(B.mantissa + rbase + 8 * ci);
                    sx[u] = __ldg(reinterpret_cast<const ulonglong2*>(sgn + kstride * (ci >> 3)));
                }
            }
#pragma unroll
            for (int u = 0; u < ROW_CHUNKS; ++u) {
                const int ci = cb + 32 * u, c0 = 8 * ci;
                if (ci >= nch) break;
                if (B.vec8) {
                    uint32_t pw[4] = {pu[u].x, pu[u].y, pu[u].z, pu[u].w};
                    uint32_t mw[4] = {mu[u].x, mu[u].y, mu[u].z, mu[u].w};
                    const uint32_t vw[4] = {vu[u].x, vu[u].y, vu[u].z, vu[u].w};
                    const unsigned gk = link_gates(sx[u], c0, rail + c0, pw, mw);
                    uint64_t sc2[4];
                    scale_pairs(sc2, rows_lanes, srow, S + c0);
                    apply8_gated(vw, pw, mw, sc2, gk, B.eff_wd, lr);
                    *reinterpret_cast<uint4*>(B.param + rbase + c0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *reinterpret_cast<uint4*>(B.mantissa + rbase + c0) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
                } else {
                    // unaligned or n % 8 != 0: element by element, the rail where the bits do not decide
                    const unsigned sw = link_bits8(sgn[kstride * (ci >> 3)], (c0 & 63) >> 2);
                    const unsigned xw = link_bits8(sgn[kstride * (ci >> 3) + 1], (c0 & 63) >> 2);
                    for (int k = 0; k < 8 && c0 + k < B.n; ++k) {
                        uint16_t pp = B.param[rbase + c0 + k], mm = B.mantissa[rbase + c0 + k];
                        const uint32_t wb = (static_cast<uint32_t>(pp) << 16) | mm;
                        const int bit = k;
                        const bool ok = (!((xw >> bit) & 1u) && (((wb >> 23) & 0xffu) - 87u) <= 167u)
                                            ? (((sw >> bit) ^ (wb >> 31)) & 1u) == 0u
                                            : __fmul_rn(rail[c0 + k], __uint_as_float(wb)) >= 0.f;
                        tail_element_gated(bf2f(B.update[rbase + c0 + k]), rows_lanes ? srow : S[c0 + k], ok, B.eff_wd,
                                           lr, pp, mm);
                        B.param[rbase + c0 + k] = pp;
                        B.mantissa[rbase + c0 + k] = mm;
                    }
                }
            }
        }
    }
}

// Blocks of the lane-power kernel resident at once on each device (cached per device).
static int g_power_blocks[64];

cudaError_t launch_tail_power(const TailParams& p, cudaStream_t stream) {
    TailParams q = p;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    int& resident = g_power_blocks[dev & 63];
    if (resident == 0) {
        int per_sm = 0, sms = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lane_power_kernel, 256, 0))) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
        resident = per_sm > 0 && sms > 0 ? per_sm * sms : 152;
    }
    // Lanes along rows: the resident blocks left beside the lanes-along-columns blocks, shared
    // between the banks by their row groups (at least one block each, at most one warp per group).
    long long col_blocks = 0, groups = 0;
    for (int i = 0; i < q.nbanks; ++i) {
        if (q.bank[i].m >= q.bank[i].n)
            groups += power_groups(q.bank[i]);
        else
            col_blocks += power_blocks(q.bank[i]);
    }
    const long long budget = resident - col_blocks > resident / 2 ? resident - col_blocks : resident / 2;
    for (int i = 0; i < q.nbanks; ++i) {
        TailBank& B = q.bank[i];
        if (B.m < B.n) continue;
        const long long gb = power_groups(B), most = (gb + 7) / 8;
        long long nb = (budget * gb + groups / 2) / groups;
        nb = nb < 1 ? 1 : (nb > most ? most : nb);
        B.power_nblk = static_cast<int>(nb);
    }
    long long blocks = 0;
    for (int i = 0; i < q.nbanks; ++i) {
        q.bank[i].power_begin = blocks;
        blocks += power_blocks(q.bank[i]);
    }
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(lane_power_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, q);
}

cudaError_t launch_tail_scale(const TailParams& p, cudaStream_t stream) {
    return launch_pdl(lane_scale_kernel, dim3(p.total_mats), dim3(SCALE_THREADS), 0, stream, p);
}

// Blocks of each apply kernel that are resident at once on this device (cached per device):
// the grid-stride loops cover the work in one wave of resident blocks, so no partial second
// wave trails the first.
static int g_apply_blocks[2][64];

cudaError_t launch_tail_apply(const TailParams& p, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    bool link = true;  // the row kernel, with the link's sign words, when every bank has them
    for (int i = 0; i < p.nbanks; ++i) link = link && p.bank[i].sign != nullptr;
    void (*kernel)(TailParams) = link ? tail_apply_rows_kernel : tail_apply_kernel;
    int& resident = g_apply_blocks[link ? 1 : 0][dev & 63];
    if (resident == 0) {
        int per_sm = 0, sms = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0))) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) return e;
        resident = per_sm > 0 && sms > 0 ? per_sm * sms : 152;
    }
    const long long work = link ? (p.total_rows + 7) / 8 : (p.total_chunks + 255) / 256;  // blocks to cover it
    long long blocks = work < resident ? work : resident;
    if (blocks < 1) blocks = 1;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
}

}  // namespace anvil
