// anvil_gemm.cu -- the three contractions of every spectral map of the ANVIL cascade
// (page "modded-nanogpt track_1_short/optim/anvil.py", anvil_cascade: the XTX / XXT,
// ba_plus_cAA and baddbmm steps), as one batched tcgen05 GEMM kernel for sm_103a:
//
//   OP_GRAM / OP_GRAM_NORM : A  = bf16(Y Y^T)            [/ d^2 for the first Gram]
//   OP_SQPOLY              : B  = bf16(b A + c A A)
//   OP_XUPDATE(_OUT)       : Y' = bf16(a Y + B Y)        [written to out for the last map]
//
// in the small-side-major layout of anvil_internal.h.  A and B are symmetric, so the
// Gram and the A A product compute only the upper-triangle 128x128 tiles and store each
// off-diagonal tile twice (itself and its mirror).  A A contracts A's rows with A's
// rows (A A = A A^T), so every operand is K-major except Y in the X-update, which is
// read MN-major (contiguous along the output columns).
//
// One CTA computes one 128x128 output tile of one matrix; the grid covers every tile
// of every matrix of up to four banks (a grouped launch).  Warp roles: warp 0 lane 0
// issues TMA loads into a STAGES-deep shared-memory ring, warp 1 lane 0 issues
// tcgen05.mma (M = 128, N = 128, K = 16) into a 128-column fp32 TMEM accumulator,
// warp 2 owns the TMEM allocation; then all four warps read the accumulator back with
// tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = tile rows) and run the fused epilogue.
// Every wait is bounded (anvil_device.cuh); a wait that gives up sets the device error
// word, the tile's epilogue is skipped, and the CTA still frees its TMEM and exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "anvil_device.cuh"
#include "anvil_internal.h"

namespace anvil {

constexpr int STAGES = 3;
constexpr int A_STAGE = TILE * BK * 2;  // 16 KB
constexpr int B_STAGE = TILE * BK * 2;  // 16 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 128;

template <int OP>
struct OpTraits {
    static constexpr bool sym = (OP == OP_GRAM || OP == OP_GRAM_NORM || OP == OP_SQPOLY);
    static constexpr bool xupdate = (OP == OP_XUPDATE || OP == OP_XUPDATE_OUT);
};

__device__ __forceinline__ void load32_bf16(const uint16_t* src, float (&f)[32]) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 u = p[v];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            f[8 * v + 2 * q] = bf2f(static_cast<uint16_t>(w[q] & 0xffffu));
            f[8 * v + 2 * q + 1] = bf2f(static_cast<uint16_t>(w[q] >> 16));
        }
    }
}

__device__ __forceinline__ void store32_bf16(uint16_t* dst, const uint16_t (&o)[32]) {
    uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = static_cast<uint32_t>(o[8 * v + 2 * q]) |
                   (static_cast<uint32_t>(o[8 * v + 2 * q + 1]) << 16);
        p[v] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int OP>
__global__ void __launch_bounds__(128) gemm_kernel(const __grid_constant__ GemmParams p) {
    using TR = OpTraits<OP>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t acc_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ int aborted;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- which tile of which matrix of which bank
    const int t = blockIdx.x;
    int bi = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (t >= p.bank[i].tile_begin) bi = i;
    const GemmBank& bk = p.bank[bi];
    const int local = t - bk.tile_begin;
    const int mat = local / bk.tiles_per_mat;
    int r = local - mat * bk.tiles_per_mat;
    int ti, tj;
    if (TR::sym) {
        ti = 0;
        while (r >= bk.T - ti) {
            r -= bk.T - ti;
            ++ti;
        }
        tj = ti + r;
    } else {
        ti = r / bk.nt_n;
        tj = r - ti * bk.nt_n;
    }

    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(&acc_bar, 1);
        fence_mbar_init();
        aborted = 0;
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&bk.tm_a);
        tma_prefetch_desc(&bk.tm_b);
    }
    if (warp == 2) tmem_alloc(&tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int nkb = bk.num_kb;
    int issued = 0;  // k-blocks whose loads the producer armed

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            const uint32_t round = kb / STAGES;
            if (!mbar_wait(&empty_bar[s], (round & 1u) ^ 1u, p.err)) {
                aborted = 1;
                break;
            }
            issued = kb + 1;
            uint8_t* sa = smem + s * STAGE_BYTES;
            uint8_t* sb = sa + A_STAGE;
            mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
            tma_load_3d(sa, &bk.tm_a, &full_bar[s], kb * BK, ti * TILE, mat);
            if (TR::xupdate) {
                // Y rows kb*64 .. +63 (the contraction index), columns tj*128 .. +127 in
                // two 64-column boxes: MN-major chunks 8 KB apart.
                tma_load_3d(sb, &bk.tm_b, &full_bar[s], tj * TILE, kb * BK, mat);
                tma_load_3d(sb + 8192, &bk.tm_b, &full_bar[s], tj * TILE + 64, kb * BK, mat);
            } else {
                tma_load_3d(sb, &bk.tm_b, &full_bar[s], kb * BK, tj * TILE, mat);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_bf16_f32(TILE, TILE, false, TR::xupdate);
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % STAGES;
            const uint32_t round = kb / STAGES;
            if (!mbar_wait(&full_bar[s], round & 1u, p.err)) {
                aborted = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + s * STAGE_BYTES);
            const uint32_t b0 = a0 + A_STAGE;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                const uint64_t bd = TR::xupdate ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                                                : smem_desc_sw128(b0 + kk * 32, 16, 1024);
                umma_bf16(tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&empty_bar[s]);  // frees the stage once these MMAs have read it
        }
        umma_commit(&acc_bar);  // accumulator complete
    }
    __syncwarp();

    // ---------------- epilogue: all four warps
    const bool acc_ok = mbar_wait(&acc_bar, 0, p.err);
    __syncthreads();  // makes the producer's / issuer's abort flag visible
    tc_fence_after();
    if (acc_ok && !aborted) {
        const int row = ti * TILE + warp * 32 + lane;  // row in the padded small side
        const size_t sq = static_cast<size_t>(bk.s_pad);
        float dd = 0.f;
        if (OP == OP_GRAM_NORM) {
            const float d = bk.d[mat];
            dd = __fmul_rn(d, d);
        }
#pragma unroll 1
        for (int cc = 0; cc < TILE / 32; ++cc) {
            float v[32];
            tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + cc * 32, v);
            const int col0 = tj * TILE + cc * 32;
            uint16_t o[32];
            if (OP == OP_GRAM) {
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = f2bf(v[q]);
            } else if (OP == OP_GRAM_NORM) {
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = f2bf(__fdiv_rn(round_bf(v[q]), dd));
            } else if (OP == OP_SQPOLY) {
                float av[32];
                load32_bf16(bk.src + (static_cast<size_t>(mat) * sq + row) * sq + col0, av);
#pragma unroll
                for (int q = 0; q < 32; ++q)
                    o[q] = f2bf(__fadd_rn(__fmul_rn(p.b, av[q]), __fmul_rn(p.c, v[q])));
            } else {
                float yv[32];
                load32_bf16(bk.src + (static_cast<size_t>(mat) * sq + row) * bk.L_pad + col0, yv);
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = f2bf(__fadd_rn(__fmul_rn(p.a, yv[q]), v[q]));
            }

            if (TR::sym) {
                uint16_t* base = bk.dst + static_cast<size_t>(mat) * sq * sq;
                store32_bf16(base + row * sq + col0, o);
                if (ti != tj) {
                    // mirror: column `row` of rows col0..col0+31; a warp writes 64 contiguous
                    // bytes per q
#pragma unroll
                    for (int q = 0; q < 32; ++q) base[(col0 + q) * sq + row] = o[q];
                }
            } else if (OP == OP_XUPDATE) {
                store32_bf16(bk.dst + (static_cast<size_t>(mat) * sq + row) * bk.L_pad + col0, o);
            } else {  // OP_XUPDATE_OUT: natural [m, n] layout, clipped to the real extent
                const int m = bk.m, n = bk.n;
                uint16_t* out = bk.dst + static_cast<size_t>(mat) * m * n;
                if (!bk.tall) {
                    if (row < m) {
                        uint16_t* dst = out + static_cast<size_t>(row) * n + col0;
                        if (col0 + 32 <= n && (n & 7) == 0 &&
                            (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
                            store32_bf16(dst, o);
                        } else {
#pragma unroll
                            for (int q = 0; q < 32; ++q)
                                if (col0 + q < n) dst[q] = o[q];
                        }
                    }
                } else if (row < n) {
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (col0 + q < m) out[static_cast<size_t>(col0 + q) * n + row] = o[q];
                }
            }
        }
    }
    if (aborted && warp == 0 && lane == 0) {
        // Let the copies still in flight land before the CTA's shared memory goes away:
        // the last load armed on each stage is that stage's latest phase.
        for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
            mbar_wait(&full_bar[kb % STAGES], (static_cast<uint32_t>(kb) / STAGES) & 1u, p.err);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) tmem_dealloc(tmem, TMEM_COLS);
}

template <int OP>
static cudaError_t launch_op(const GemmParams& p, cudaStream_t stream) {
    gemm_kernel<OP><<<p.total_tiles, 128, GEMM_SMEM, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(GemmOp op, const GemmParams& p, cudaStream_t stream) {
    if (p.total_tiles <= 0) return cudaSuccess;
    switch (op) {
        case OP_GRAM: return launch_op<OP_GRAM>(p, stream);
        case OP_GRAM_NORM: return launch_op<OP_GRAM_NORM>(p, stream);
        case OP_SQPOLY: return launch_op<OP_SQPOLY>(p, stream);
        case OP_XUPDATE: return launch_op<OP_XUPDATE>(p, stream);
        case OP_XUPDATE_OUT: return launch_op<OP_XUPDATE_OUT>(p, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t gemm_prepare() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<OP_GRAM>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM))) return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<OP_GRAM_NORM>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM))) return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<OP_SQPOLY>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM))) return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<OP_XUPDATE>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM))) return e;
    if ((e = cudaFuncSetAttribute(gemm_kernel<OP_XUPDATE_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM))) return e;
    return cudaSuccess;
}

}  // namespace anvil
