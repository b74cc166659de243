// issue_probe.cu -- a diagnostic program (not part of libanvil): the rate at which one
// thread can keep the 2-SM tensor pipe busy, in SM cycles per 64-deep k-block of
// 256 x 256 tiles (four tcgen05.mma.cta_group::2 of K = 16), on 76 CTA pairs at once.
//
//   chain       operands fixed in shared memory, one MMA chain, a commit per k-block:
//               the tensor pipe's own rate
//   chain+N     the same with N dependent integer adds per k-block on the issuing
//               thread: how much of a k-block the thread has to spare
//   ring/block  operands streamed by TMA from a 380 MB bf16 buffer through a 5-stage ring
//               (one producer thread per CTA), 44-k-block tiles into two alternating
//               accumulators, an epilogue warpgroup reading each finished accumulator;
//               the issuer waits (blocking) for each stage's barrier before its MMAs
//   ring/piped  the same, but the issuer tests the next stage's barrier (without
//               blocking) after issuing the current k-block's MMAs, and waits only when
//               that test failed
//   .../lean    the ring cases with each MMA's descriptors formed from a per-k-block low
//               word and the constant high word (sw128_desc) instead of the full helper
//
// Every wait is bounded (anvil_device.cuh); a wait that gives up sets the error word,
// which the program prints.  Usage: issue_probe  (prints one line per case)
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <algorithm>
#include <vector>

#include "anvil_device.cuh"

using namespace anvil;

namespace {

constexpr int STAGES = 5;
constexpr int BOX = 128 * 64 * 2;  // one CTA's 128 rows x 64 columns of bf16 (16 KB)
constexpr int STG = 2 * BOX;       // A rows and B columns of one k-block
constexpr int ROWS = 768, COLS = 2816, MATS = 88;
constexpr int NKB = COLS / 64;

enum Mode : int { CHAIN = 0, RING_BLOCKING = 1, RING_PIPED = 2 };

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }

template <int MODE, bool LEAN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
probe_kernel(const __grid_constant__ CUtensorMap tm, int chain_kb, int adds, int ntiles, unsigned long long* out,
             unsigned* err) {
    constexpr int mode = MODE;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], done;
    __shared__ uint32_t slot;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);  // four epilogue warps in each CTA
        }
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    // a fixed operand pattern for the chain cases: +-(1 + m/128) * 2^-7
    for (int i = threadIdx.x; i < STG / 4; i += blockDim.x) {
        const uint32_t h = static_cast<uint32_t>(i) * 2654435761u;
        const uint32_t lo = 0x3c00u | (h & 0x7fu) | ((h >> 7) & 1u) << 15;
        const uint32_t hi = 0x3c00u | ((h >> 8) & 0x7fu) | ((h >> 15) & 1u) << 15;
        reinterpret_cast<uint32_t*>(smem)[i] = lo | (hi << 16);
    }
    fence_proxy_async_smem();
    if (warp == 1) tmem_alloc_pair(&slot, 512);
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = slot;
    const uint32_t idesc = idesc_bf16_f32(256, 256, false, false);

    if (mode == CHAIN) {
        if (warp == 1 && lane == 0 && rank == 0) {
            const uint32_t a0 = smem_u32(smem), b0 = a0 + BOX;
            uint32_t junk = 0;
            const unsigned long long t0 = clock64();
            for (int kb = 0; kb < chain_kb; ++kb) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16_pair(tmem, kdesc(a0 + kk * 32), kdesc(b0 + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                umma_commit_pair(&empty[kb % STAGES], 3);
                for (int e = 0; e < adds; ++e) asm volatile("add.u32 %0, %0, %1;" : "+r"(junk) : "r"(kb));
            }
            umma_commit_pair(&done, 3);
            mbar_wait(&done, 0, err);
            out[2 * pair] = clock64() - t0;
            out[2 * pair + 1] = static_cast<unsigned long long>(chain_kb);
            if (junk == 0x9e3779b9u) out[2 * npairs] = junk;  // keeps the adds
        } else if (warp == 1 && lane == 0) {
            mbar_wait(&done, 0, err);
        }
    } else if (warp == 0 && lane == 0) {
        // producer: both CTAs load their halves, completing on the leader's barrier
        int it = 0;
        bool ok = true;
        for (int t = pair; t < ntiles && ok; t += npairs) {
            const int mat = (t / 9) % MATS, bi = (t % 9) / 3, bj = t % 3;
            for (int kb = 0; kb < NKB; ++kb, ++it) {
                const int s = it % STAGES;
                if (!mbar_wait(&empty[s], static_cast<uint32_t>((it / STAGES) & 1) ^ 1u, err)) {
                    ok = false;
                    break;
                }
                if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * STG);
                const uint32_t fb = map_to_rank(&full[s], 0);
                uint8_t* sa = smem + s * STG;
                tma_load_3d_pair(sa, &tm, fb, kb * 64, bi * 256 + 128 * static_cast<int>(rank), mat);
                tma_load_3d_pair(sa + BOX, &tm, fb, kb * 64, bj * 256 + 128 * static_cast<int>(rank), mat);
            }
        }
        if (rank == 0)  // the last loads land before the CTA may leave
            for (int k = it - STAGES < 0 ? 0 : it - STAGES; k < it; ++k)
                mbar_wait(&full[k % STAGES], static_cast<uint32_t>((k / STAGES) & 1), err);
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // MMA issuer
        const uint32_t stage0 = smem_u32(smem);
        int s = 0, mt = 0;
        uint32_t ph = 0;
        bool ready = false, ok = true;
        long long nkb = 0;
        const unsigned long long t0 = clock64();
        for (int t = pair; t < ntiles && ok; t += npairs, ++mt) {
            const int ab = mt & 1;
            if (!mbar_wait(&tempty[ab], static_cast<uint32_t>((mt >> 1) & 1) ^ 1u, err)) break;
            tc_fence_after();
            const uint32_t dacc = tmem + static_cast<uint32_t>(ab * 256);
            for (int kb = 0; kb < NKB; ++kb) {
                if (!(mode == RING_PIPED && ready) && !mbar_wait(&full[s], ph, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = stage0 + static_cast<uint32_t>(s * STG), b0 = a0 + BOX;
                const uint32_t a_lo = sw128_desc_lo(a0, 16), b_lo = sw128_desc_lo(b0, 16);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (LEAN)
                        umma_bf16_pair(dacc, sw128_desc(a_lo + kk * 2), sw128_desc(b_lo + kk * 2), idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    else
                        umma_bf16_pair(dacc, kdesc(a0 + kk * 32), kdesc(b0 + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
                }
                const int s_next = s + 1 == STAGES ? 0 : s + 1;
                const uint32_t ph_next = s_next == 0 ? ph ^ 1u : ph;
                if (mode == RING_PIPED) ready = mbar_test_wait(smem_u32(&full[s_next]), ph_next);
                umma_commit_pair(&empty[s], 3);
                s = s_next;
                ph = ph_next;
                ++nkb;
            }
            if (ok) umma_commit_pair(&tfull[ab], 3);
        }
        umma_commit_pair(&done, 3);
        mbar_wait(&done, 0, err);
        out[2 * pair] = clock64() - t0;
        out[2 * pair + 1] = static_cast<unsigned long long>(nkb);
    } else if (warp == 1 && lane == 0) {
        mbar_wait(&done, 0, err);
    } else if (warp >= 2) {
        // epilogue warpgroup: read each finished accumulator, then free it
        const uint32_t quad = static_cast<uint32_t>((warp & 3) * 32) << 16;
        float acc = 0.f;
        int mt = 0;
        for (int t = pair; t < ntiles; t += npairs, ++mt) {
            const int ab = mt & 1;
            if (!mbar_wait(&tfull[ab], static_cast<uint32_t>((mt >> 1) & 1), err)) break;
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                float v[32];
                tmem_ld_32x32b_x32(tmem + quad + static_cast<uint32_t>(ab * 256 + j * 32), v);
                acc += v[0] + v[31];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(&tempty[ab], 0));
        }
        if (acc == 1234.5f) out[2 * npairs] = 1;  // keeps the reads
    }
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

__global__ void fill_kernel(uint32_t* p, size_t n) {
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x) {
        const uint32_t h = static_cast<uint32_t>(i) * 2246822519u;
        p[i] = (0x3c00u | (h & 0x7fu)) | ((0x3c00u | ((h >> 8) & 0x7fu)) << 16);
    }
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

int main() {
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) {
        printf("issue_probe needs an sm_103 device\n");
        return 1;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) || !fn) {
        printf("no tensor-map encoder\n");
        return 1;
    }
    const size_t bytes = size_t(MATS) * ROWS * COLS * 2;
    void* buf = nullptr;
    unsigned long long* d_out = nullptr;
    unsigned* d_err = nullptr;
    const int npairs = sms / 2;
    if (cudaMalloc(&buf, bytes) || cudaMalloc(&d_out, sizeof(unsigned long long) * (2 * npairs + 1)) ||
        cudaMalloc(&d_err, sizeof(unsigned))) {
        printf("allocation failed\n");
        return 1;
    }
    cudaMemset(d_err, 0, sizeof(unsigned));
    fill_kernel<<<1024, 256>>>(static_cast<uint32_t*>(buf), bytes / 4);
    CUtensorMap tm;
    const cuuint64_t dims[3] = {COLS, ROWS, MATS};
    const cuuint64_t strides[2] = {cuuint64_t(COLS) * 2, cuuint64_t(ROWS) * COLS * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (reinterpret_cast<EncodeFn>(fn)(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, buf, dims, strides, box, estr,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS) {
        printf("tensor map encoding failed\n");
        return 1;
    }
    const int smem = STAGES * STG + 1024;
    typedef void (*Kernel)(const CUtensorMap, int, int, int, unsigned long long*, unsigned*);
    struct Case {
        const char* name;
        Kernel k;
        int adds;
    };
    const Case cases[] = {{"chain", probe_kernel<CHAIN, false>, 0},
                          {"chain+32", probe_kernel<CHAIN, false>, 32},
                          {"chain+64", probe_kernel<CHAIN, false>, 64},
                          {"chain+128", probe_kernel<CHAIN, false>, 128},
                          {"ring/block", probe_kernel<RING_BLOCKING, false>, 0},
                          {"ring/piped", probe_kernel<RING_PIPED, false>, 0},
                          {"ring/block/lean", probe_kernel<RING_BLOCKING, true>, 0},
                          {"ring/piped/lean", probe_kernel<RING_PIPED, true>, 0}};
    for (const Case& c : cases) cudaFuncSetAttribute(c.k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const int ntiles = MATS * 9;  // every 256 x 256 block of every matrix, K = 2816
    printf("| case | SM cycles per 64-deep k-block (median CTA pair) |\n|---|---|\n");
    for (const Case& c : cases) {
        double med = 0.0;
        for (int rep = 0; rep < 3; ++rep) {
            c.k<<<2 * npairs, 192, smem>>>(tm, 2000, c.adds, ntiles, d_out, d_err);
            if (cudaDeviceSynchronize() != cudaSuccess) {
                printf("launch failed: %s\n", cudaGetErrorString(cudaGetLastError()));
                return 1;
            }
            std::vector<unsigned long long> h(2 * npairs);
            cudaMemcpy(h.data(), d_out, sizeof(unsigned long long) * 2 * npairs, cudaMemcpyDeviceToHost);
            std::vector<double> per;
            for (int i = 0; i < npairs; ++i)
                if (h[2 * i + 1]) per.push_back(double(h[2 * i]) / double(h[2 * i + 1]));
            std::sort(per.begin(), per.end());
            if (rep == 2 && !per.empty()) med = per[per.size() / 2];
        }
        printf("| %s | %.1f |\n", c.name, med);
    }
    unsigned err = 0;
    cudaMemcpy(&err, d_err, sizeof(unsigned), cudaMemcpyDeviceToHost);
    printf("\nerror word %u\n", err);
    return err ? 1 : 0;
}
