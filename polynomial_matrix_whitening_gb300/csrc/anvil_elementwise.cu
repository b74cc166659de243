// anvil_elementwise.cu -- the HBM-bound kernels of the ANVIL bank step:
//   * momentum_kernel: twin-rail Nesterov momentum + bf16 cast (page "modded-nanogpt
//     track_1_short/optim/anvil.py", anvil_cascade, first block), writing X in the
//     small-side-major working layout and the per-64-block sums of squares of the bf16
//     values, from which the first Gram's diagonal (hence the trace) is read;
//   * norm_d_kernel: d = sqrt(tr) * FROBENIUS_MARGIN + FROBENIUS_EPS per matrix;
//   * normalize_kernel: the normalised X = bf16(X / d), streamed at HBM rate;
//   * extraction kernels for the traced (parity-test) path and the wait self-test.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "anvil_device.cuh"
#include "anvil_internal.h"

namespace anvil {

__device__ unsigned g_error_word;

// One 64x64 tile of the padded natural extent of one matrix per block, 256 threads.
// Thread (tx, ty) = (tid % 16, tid / 16) handles columns c0 + 4 tx .. +3 of rows
// r0 + ty + 16 k, k = 0..3.  Every rounding matches the page's fp32 tensor ops one
// operation at a time (no fused multiply-add): lerp(s, e, w) = s + w (e - s).
__global__ void __launch_bounds__(256) momentum_kernel(const __grid_constant__ MomentumParams p) {
    __shared__ __align__(16) uint16_t tileT[64][64 + 8];  // tall: [s-index][L-index]
    pdl_allow_next();
    pdl_wait_previous();

    const int t = blockIdx.x;
    int bi = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (t >= p.bank[i].tile_begin) bi = i;
    const MomentumBank& B = p.bank[bi];
    const int local = t - B.tile_begin;
    const int per_mat = B.tiles_r * B.tiles_c;
    const int mat = local / per_mat;
    const int rem = local - mat * per_mat;
    const int tr = rem / B.tiles_c, tc = rem - (rem / B.tiles_c) * B.tiles_c;
    const int r0 = tr * 64, c0 = tc * 64;

    float mom = B.momentum, fbeta = B.fast_beta, fw = B.fast_weight, sbeta = B.slow_beta;
    if (p.dev_scalars) {
        const float* s = p.dev_scalars + 4 * bi;
        mom = s[0];
        fbeta = s[1];
        fw = s[2];
        sbeta = s[3];
    }
    const float wf = __fsub_rn(1.0f, fbeta);
    const float ws = __fsub_rn(1.0f, sbeta);
    const float omw = __fsub_rn(1.0f, fw);

    const int m = B.m, n = B.n;
    const size_t mn = static_cast<size_t>(m) * n;
    const float* G = static_cast<const float*>(B.grad) + static_cast<size_t>(mat) * mn;
    const uint16_t* Gh = static_cast<const uint16_t*>(B.grad) + static_cast<size_t>(mat) * mn;
    float* V0 = B.velocity + static_cast<size_t>(mat) * mn;
    float* V1 = V0 + static_cast<size_t>(B.g) * mn;
    uint16_t* Y = B.y + static_cast<size_t>(mat) * B.s_pad * B.L_pad;
    float* part = B.part + static_cast<size_t>(mat) * B.nlb * B.s_pad;

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int c = c0 + 4 * tx;

#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = r0 + ty + 16 * k;
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        // tail link: the new slow rail's sign, and whether the tail must read the value
        bool sgn[4] = {false, false, false, false}, exq[4] = {true, true, true, true};
        if (r < m) {
            const size_t base = static_cast<size_t>(r) * n + c;
            float g[4] = {0.f, 0.f, 0.f, 0.f}, v0[4] = {0.f, 0.f, 0.f, 0.f}, v1[4] = {0.f, 0.f, 0.f, 0.f};
            bool in[4];
            if (B.vec4) {
                const bool row_in = c < n;  // n % 4 == 0: all four or none
                if (row_in) {
                    float4 g4;
                    if (B.grad_bf16) {
                        const uint2 h = __ldcs(reinterpret_cast<const uint2*>(Gh + base));
                        g4 = make_float4(bf2f(static_cast<uint16_t>(h.x & 0xffffu)), bf2f(static_cast<uint16_t>(h.x >> 16)),
                                         bf2f(static_cast<uint16_t>(h.y & 0xffffu)), bf2f(static_cast<uint16_t>(h.y >> 16)));
                    } else {
                        g4 = __ldcs(reinterpret_cast<const float4*>(G + base));
                    }
                    const float4 a4 = __ldcs(reinterpret_cast<const float4*>(V0 + base));
                    const float4 b4 = __ldcs(reinterpret_cast<const float4*>(V1 + base));
                    g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
                    v0[0] = a4.x; v0[1] = a4.y; v0[2] = a4.z; v0[3] = a4.w;
                    v1[0] = b4.x; v1[1] = b4.y; v1[2] = b4.z; v1[3] = b4.w;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) in[q] = row_in;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    in[q] = c + q < n;
                    g[q] = in[q] ? (B.grad_bf16 ? bf2f(Gh[base + q]) : G[base + q]) : 0.f;
                    v0[q] = in[q] ? V0[base + q] : 0.f;
                    v1[q] = in[q] ? V1[base + q] : 0.f;
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = __fadd_rn(v0[q], __fmul_rn(wf, __fsub_rn(g[q], v0[q])));
                const float b = __fadd_rn(v1[q], __fmul_rn(ws, __fsub_rn(g[q], v1[q])));
                v0[q] = a;
                v1[q] = b;
                const float blend = __fadd_rn(__fmul_rn(fw, a), __fmul_rn(omw, b));
                const float y = __fadd_rn(g[q], __fmul_rn(mom, __fsub_rn(blend, g[q])));
                x[q] = in[q] ? round_bf(y) : 0.f;
                sgn[q] = in[q] && signbit(b);
                exq[q] = !in[q] || !(fabsf(b) >= 0x1p-100f && fabsf(b) <= 3.402823466e38f);
            }
            if (B.vec4) {
                if (in[0]) {
                    __stcs(reinterpret_cast<float4*>(V0 + base), make_float4(v0[0], v0[1], v0[2], v0[3]));
                    __stcs(reinterpret_cast<float4*>(V1 + base), make_float4(v1[0], v1[1], v1[2], v1[3]));
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (in[q]) {
                        V0[base + q] = v0[q];
                        V1[base + q] = v1[q];
                    }
            }
        }
        if (B.gate) {
            // sign and exact-read bits of the warp's two rows (lanes 0-15: row of the even
            // ty, 16-31: the odd one): bit 16 q + tx of a row's word is column c0 + 4 tx + q
            const int half = threadIdx.x & 16;
            uint64_t sw = 0, xw = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const unsigned bs = __ballot_sync(0xffffffffu, sgn[q]);
                const unsigned bx = __ballot_sync(0xffffffffu, exq[q]);
                sw |= static_cast<uint64_t>((bs >> half) & 0xffffu) << (16 * q);
                xw |= static_cast<uint64_t>((bx >> half) & 0xffffu) << (16 * q);
            }
            if (tx == 0 && r < m && c0 < n) {
                // [g, nck, m, 2]: a tile's 64 rows of one column chunk are 1 KB contiguous
                uint64_t* gw = B.gate + ((static_cast<size_t>(mat) * B.nck + tc) * m + r) * 2;
                *reinterpret_cast<ulonglong2*>(gw) = make_ulonglong2(sw, xw);
            }
        }
        if (!B.tall) {
            // wide: Y = X, row r, columns c..c+3 (inside the padded extent by construction)
            uint2 pk;
            pk.x = static_cast<uint32_t>(f2bf(x[0])) | (static_cast<uint32_t>(f2bf(x[1])) << 16);
            pk.y = static_cast<uint32_t>(f2bf(x[2])) | (static_cast<uint32_t>(f2bf(x[3])) << 16);
            *reinterpret_cast<uint2*>(Y + static_cast<size_t>(r) * B.L_pad + c) = pk;
            // sum of squares of this row over the tile's 64 columns (16 lanes share a row)
            float sq = __fadd_rn(__fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1])),
                                 __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3])));
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, off));
            if (tx == 0) part[static_cast<size_t>(tc) * B.s_pad + r] = sq;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) tileT[4 * tx + q][ty + 16 * k] = f2bf(x[q]);
        }
    }
    if (B.tall) {
        __syncthreads();
        // tall: Y = X^T; Y row (c0 + cl) gets the 64 L-indices r0 .. r0+63 of this tile
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int cl = ty + 16 * k;
            const uint2 pk = *reinterpret_cast<const uint2*>(&tileT[cl][4 * tx]);
            *reinterpret_cast<uint2*>(Y + static_cast<size_t>(c0 + cl) * B.L_pad + r0 + 4 * tx) = pk;
        }
        // sum of squares of each s-index over the tile's 64 L-indices: 4 threads per index
        const int cl = threadIdx.x >> 2, qq = threadIdx.x & 3;
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float v = bf2f(tileT[cl][16 * qq + j]);
            sq = __fadd_rn(sq, __fmul_rn(v, v));
        }
        sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, 1));
        sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, 2));
        if (qq == 0) part[static_cast<size_t>(tr) * B.s_pad + c0 + cl] = sq;
    }
}

// The step's first kernel is launched without programmatic serialisation, so it starts
// after whatever the stream ran before it has finished.  Measured on a CUDA graph of 20
// consecutive steps: with a programmatic edge from the previous step's cascade the steps
// took 1.11-1.13 ms, with a plain edge 1.05-1.07 ms, as separate per-step graphs do.
// (Its griddepcontrol.wait is then a no-op; its launch_dependents still lets the norm_d
// kernel that follows be scheduled early.)
cudaError_t launch_momentum(const MomentumParams& p, cudaStream_t stream) {
    momentum_kernel<<<dim3(p.total_tiles), dim3(256), 0, stream>>>(p);
    return cudaGetLastError();
}

static_assert(SCHED_COUNTERS <= 256, "norm_d_kernel zeroes the item counters with one block");

// One block per matrix.  Diagonal entry i of the first Gram is the fp32 sum of the
// squares of row i of Y (the momentum kernel's per-64-column partials, summed here in
// column-block order), rounded to bf16 as the page stores the Gram; the trace sums those
// in fp32 (a fixed order: per thread, then per warp by shuffles, then over the warps).
// A thread's partial loads go out eight at a time, so a row costs a few memory round
// trips rather than one per column block.
constexpr int NORM_THREADS = 1024;
__global__ void __launch_bounds__(NORM_THREADS) norm_d_kernel(const __grid_constant__ NormParams p) {
    __shared__ float red[NORM_THREADS / 32];
    pdl_allow_next();
    pdl_wait_previous();
    const int gm = blockIdx.x;
    int bi = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (gm >= p.bank[i].mat_begin) bi = i;
    const NormBank& B = p.bank[bi];
    const int lm = gm - B.mat_begin;
    if (threadIdx.x == 0) p.counters[gm] = 0u;
    if (gm == 0 && threadIdx.x < SCHED_COUNTERS) p.counters[p.total_mats + threadIdx.x] = 0u;
    const float* part = B.part + static_cast<size_t>(lm) * B.nlb * B.s_pad;  // [nlb][s_pad]
    float acc = 0.f;
    for (int i = threadIdx.x; i < B.s_pad; i += NORM_THREADS) {
        const float* col = part + i;
        float s = 0.f;
        int lb = 0;
        for (; lb + 8 <= B.nlb; lb += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = col[static_cast<size_t>(lb + u) * B.s_pad];
#pragma unroll
            for (int u = 0; u < 8; ++u) s = __fadd_rn(s, v[u]);
        }
        for (; lb < B.nlb; ++lb) s = __fadd_rn(s, col[static_cast<size_t>(lb) * B.s_pad]);
        acc = __fadd_rn(acc, round_bf(s));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        float w = red[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, o));
        if (threadIdx.x == 0) p.d[gm] = __fadd_rn(__fmul_rn(__fsqrt_rn(w), p.margin), p.eps);
    }
}

cudaError_t launch_norm_d(const NormParams& p, cudaStream_t stream) {
    return launch_pdl(norm_d_kernel, dim3(p.total_mats), dim3(NORM_THREADS), 0, stream, p);
}

// X / d (page "modded-nanogpt track_1_short/optim/anvil.py", anvil_cascade, the division
// of X by its normaliser) over the padded working layout, which is contiguous per bank:
// chunk k of a bank is elements 8k .. 8k + 7 of its Y0 and Y1.  A block converts
// NX_BLOCK_CHUNKS chunks of one matrix, so its bank, matrix and d are found once; each
// thread converts NX_CHUNKS of them, every load in flight before the first store, a warp's
// loads covering 32 consecutive chunks (512 bytes).  The quotient is bf16(RN(x / d)), each
// element rounded as the page's fp32 division then its bf16 cast (div4_to_bf2); the
// padding stays zero.
constexpr int NX_THREADS = 256;
constexpr int NX_CHUNKS = NX_BLOCK_CHUNKS / NX_THREADS;
__global__ void __launch_bounds__(NX_THREADS) normalize_kernel(const __grid_constant__ NormXParams p) {
    pdl_allow_next();
    pdl_wait_previous();  // d (norm_d) and X_raw (momentum)
    int b = 0;
#pragma unroll 1
    for (int k = 1; k < p.nbanks; ++k)
        if (static_cast<int>(blockIdx.x) >= p.bank[k].block_begin) b = k;
    const NormXBank& B = p.bank[b];
    const int lb = static_cast<int>(blockIdx.x) - B.block_begin;
    const float d = B.d[lb / B.blocks_per_mat];
    const float rcp = __frcp_rn(d);
    const uint64_t rcp2 = f2_pack(rcp, rcp);
    const size_t c0 = static_cast<size_t>(lb) * NX_BLOCK_CHUNKS + threadIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(B.y0) + c0;
    uint4* dst = reinterpret_cast<uint4*>(B.y1) + c0;
    uint4 v[NX_CHUNKS];
#pragma unroll
    for (int i = 0; i < NX_CHUNKS; ++i) v[i] = __ldg(src + i * NX_THREADS);
#pragma unroll
    for (int i = 0; i < NX_CHUNKS; ++i)
        dst[i * NX_THREADS] = div4_to_bf2(bf2_to_f2(v[i].x), bf2_to_f2(v[i].y), bf2_to_f2(v[i].z),
                                          bf2_to_f2(v[i].w), rcp2, d);
}

cudaError_t launch_normalize(const NormXParams& p, cudaStream_t stream) {
    if (p.total_blocks <= 0) return cudaSuccess;
    return launch_pdl(normalize_kernel, dim3(static_cast<unsigned>(p.total_blocks)), dim3(NX_THREADS), 0, stream, p);
}

// ---------------------------------------------------------------- tracing
__global__ void extract_x_kernel(const uint16_t* __restrict__ y, uint16_t* __restrict__ dst, int g,
                                 int m, int n, int tall, int s_pad, int L_pad) {
    const long long total = static_cast<long long>(g) * m * n;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(e % n);
        const int r = static_cast<int>((e / n) % m);
        const int mat = static_cast<int>(e / (static_cast<long long>(m) * n));
        const int i = tall ? c : r, l = tall ? r : c;
        dst[e] = y[(static_cast<size_t>(mat) * s_pad + i) * L_pad + l];
    }
}

cudaError_t launch_extract_x(const uint16_t* y, uint16_t* dst, int g, int m, int n, int tall,
                             int s_pad, int L_pad, cudaStream_t stream) {
    extract_x_kernel<<<1024, 256, 0, stream>>>(y, dst, g, m, n, tall, s_pad, L_pad);
    return cudaGetLastError();
}

__global__ void extract_sq_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                  int g, int s, int s_pad) {
    const long long total = static_cast<long long>(g) * s * s;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        int j = static_cast<int>(e % s);
        int i = static_cast<int>((e / s) % s);
        const int mat = static_cast<int>(e / (static_cast<long long>(s) * s));
        if (i / 256 > j / 256) {  // only the diagonal and upper 256-blocks are stored
            const int t = i;
            i = j;
            j = t;
        }
        dst[e] = src[(static_cast<size_t>(mat) * s_pad + i) * s_pad + j];
    }
}

cudaError_t launch_extract_sq(const uint16_t* src, uint16_t* dst, int g, int s, int s_pad,
                              cudaStream_t stream) {
    extract_sq_kernel<<<1024, 256, 0, stream>>>(src, dst, g, s, s_pad);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- bounded-wait self-test
// Waits on an mbarrier that nothing ever completes; the bounded wait gives up after
// limit_ns, records DEVERR_TIMEOUT and the kernel returns normally.
__global__ void wait_selftest_kernel(unsigned long long limit_ns, unsigned* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err, limit_ns);
    __syncthreads();
}

cudaError_t launch_wait_selftest(unsigned timeout_us, unsigned* err, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(timeout_us) * 1000ull,
                                               err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- per-stream error read
// Each read takes the error word with one atomic (exchange with 0 when clearing) into a
// slot of its own, which the host then copies back on the same stream.
constexpr int ERROR_SLOTS = 64;
__device__ unsigned g_error_taken[ERROR_SLOTS];

__global__ void take_error_kernel(unsigned* err, unsigned* slot, int clear) {
    *slot = clear ? atomicExch(err, 0u) : atomicOr(err, 0u);
}

cudaError_t read_error_word_on_stream(unsigned* err, int clear, unsigned* word, cudaStream_t stream) {
    static std::atomic<unsigned> next{0};
    unsigned* slots = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&slots), g_error_taken);
    if (e) return e;
    unsigned* slot = slots + (next.fetch_add(1u) % ERROR_SLOTS);
    take_error_kernel<<<1, 1, 0, stream>>>(err, slot, clear);
    if ((e = cudaGetLastError())) return e;
    if ((e = cudaMemcpyAsync(word, slot, sizeof(unsigned), cudaMemcpyDeviceToHost, stream))) return e;
    return cudaStreamSynchronize(stream);
}

unsigned* device_error_word() {
    static unsigned* cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!cache[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned*>(ptr);
    }
    return cache[dev];
}

}  // namespace anvil
