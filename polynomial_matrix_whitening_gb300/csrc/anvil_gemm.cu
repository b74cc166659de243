// anvil_gemm.cu -- the three contractions of every spectral map of the ANVIL cascade
// (page "modded-nanogpt track_1_short/optim/anvil.py", anvil_cascade: the XTX / XXT,
// ba_plus_cAA and baddbmm steps), as one batched tcgen05 GEMM kernel for sm_103a:
//
//   OP_GRAM / OP_GRAM_NORM : A  = bf16(Y Y^T)            [/ d^2 for the first Gram]
//   OP_SQPOLY              : B  = bf16(b A + c A A)
//   OP_XUPDATE(_OUT)       : Y' = bf16(a Y + B Y)        [written to out for the last map]
//
// in the small-side-major layout of anvil_internal.h.  A and B are symmetric, so the
// Gram and the A A product compute only the upper-triangle 256x256 tiles and store each
// off-diagonal tile twice (itself and its mirror).  A A contracts A's rows with A's
// rows (A A = A A^T), so every operand is K-major except Y in the X-update, which is
// read MN-major (contiguous along the output columns).
//
// CTA pairs: the kernel runs in clusters of two CTAs on two SMs; each pair computes one
// 256x256 output tile with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16).  CTA
// rank r of the pair loads rows 128r..128r+127 of the tile's A operand and columns
// 128r..128r+127 of its B operand, and holds output rows 128r.. in its own TMEM, so
// each SM streams 32 KB of operands per 64-deep k-block for 2 x 128 x 256 x 64 MACs.
// Persistent and warp-specialised: each pair walks output tiles in a snake order over
// every matrix of up to four banks (heaviest bank first).  Warp 0 (one lane) issues TMA
// loads into a STAGES-deep shared-memory ring, counted on the leader CTA's barrier;
// warp 1 owns the TMEM allocation (in both CTAs) and, in the leader CTA only, issues the
// MMAs into one of two 256-column fp32 accumulators and commits to both CTAs' barriers;
// warps 2-5 of each CTA read the other accumulator back with tcgen05.ld (warp w owns
// TMEM lanes 32 (w % 4) ..) and run the fused epilogue, so a tile's epilogue overlaps
// the next tile's MMAs.
//
// The epilogue works by quarters of 64 output columns through two shared-memory
// staging buffers: the epilogue input (A for sqpoly, Y for the X-update) arrives by
// TMA into a 128x64 box (128-byte swizzle, conflict-free 16-byte reads), the result
// is written back in place and leaves by TMA store; a transposed 64x128 box carries
// the mirror tile of the symmetric products (and the last X-update of a tall bank,
// whose output is X = Y^T).  The last X-update of a bank whose column count is not a
// multiple of 8 writes `out` with plain bounds-checked stores instead.
//
// Every wait is bounded (anvil_device.cuh): a wait that gives up sets the device error
// word and an abort flag; all roles stop, in-flight copies and MMAs are waited for
// (bounded), the TMEM is freed and the CTA exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "anvil_device.cuh"
#include "anvil_internal.h"

namespace anvil {

constexpr int SMEM_MAX = 227 * 1024;  // opt-in dynamic shared memory per block
constexpr int QBOX = TILE * 64 * 2;   // one 128 x 64 bf16 staging box (16 KB)
constexpr int EPI_GROUPS = 2;         // epilogue warp groups, one per half of the columns

template <int OP>
struct OpTraits {
    static constexpr bool sym = (OP == OP_GRAM || OP == OP_GRAM_NORM || OP == OP_SQPOLY);
    static constexpr bool xupdate = (OP == OP_XUPDATE || OP == OP_XUPDATE_OUT);
    static constexpr bool has_in = (OP == OP_SQPOLY) || xupdate;   // epilogue reads a tile
    static constexpr bool has_t = sym || OP == OP_XUPDATE_OUT;     // transposed staging box
    static constexpr int BN = PAIR;                                // output columns per CTA
    static constexpr int NQ = BN / 64;                             // quarters per tile
    static constexpr int A_STAGE = TILE * BK * 2;                  // 16 KB: this CTA's A rows
    static constexpr int B_STAGE = TILE * BK * 2;                  // 16 KB: this CTA's B half
    static constexpr int STAGE = A_STAGE + B_STAGE;
    // staging boxes (16 KB each): ops with an input stage the whole tile's input (one box
    // per quarter, loaded as soon as the epilogue starts the tile) and update it in place;
    // the Gram has one output box per epilogue group; mirrored / transposed outputs add
    // one transposed box per group.
    static constexpr int NDIR = has_in ? NQ : EPI_GROUPS;
    static constexpr int NT = has_t ? EPI_GROUPS : 0;
    static constexpr int STAGING = (NDIR + NT) * QBOX;
    static constexpr int STAGES = (SMEM_MAX - 2048 - STAGING) / STAGE;
    static constexpr int SMEM = STAGES * STAGE + STAGING + 1024;   // + alignment slack
    static constexpr uint32_t TMEM_COLS = 2 * BN;                  // two accumulators
};

// warp 0: TMA producer; warp 1: TMEM owner and MMA issuer; warps 2-9: epilogue, in two
// groups of four (one warp per TMEM lane quadrant), group h owning quarters 2h, 2h+1.
constexpr int GEMM_THREADS = 64 + EPI_GROUPS * 128;

__device__ __forceinline__ void load32_bf16(const uint16_t* src, float (&f)[32]) {
    const uint4* p = reinterpret_cast<const uint4*>(src);
    uint4 u[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) u[v] = p[v];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint32_t w[4] = {u[v].x, u[v].y, u[v].z, u[v].w};
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

struct TileCoord {
    int bi, mat, ti, tj;
};

// The k-th tile of pair c in a persistent grid of G pairs: tiles are handed out in rounds
// of G, alternating direction (a snake), so the heavy tiles at the front of the order
// spread evenly.  Returns >= total when the pair has no k-th tile.
__device__ __forceinline__ int snake_tile(int k, int c, int G) {
    return k * G + ((k & 1) ? (G - 1 - c) : c);
}

// Tile t of the grouped launch -> (bank, matrix, row block, column block), in 256s.
template <int OP>
__device__ __forceinline__ TileCoord decode_tile(const GemmParams& p, int t) {
    TileCoord c;
    c.bi = 0;
#pragma unroll 1
    for (int i = 1; i < p.nbanks; ++i)
        if (t >= p.bank[i].tile_begin) c.bi = i;
    const GemmBank& bk = p.bank[c.bi];
    const int local = t - bk.tile_begin;
    c.mat = local / bk.tiles_per_mat;
    int r = local - c.mat * bk.tiles_per_mat;
    if (OpTraits<OP>::sym) {
        c.ti = 0;
        while (r >= bk.T - c.ti) {
            r -= bk.T - c.ti;
            ++c.ti;
        }
        c.tj = c.ti + r;
    } else {
        c.ti = r / bk.nt_n;
        c.tj = r - c.ti * bk.nt_n;
    }
    return c;
}

// The elementwise part of each op's epilogue, on fp32 accumulator value v and (where
// the op has one) the bf16 input value x at the same position.
template <int OP>
__device__ __forceinline__ uint16_t epi_value(const GemmParams& p, float v, float x, float dd) {
    if (OP == OP_GRAM) return f2bf(v);
    if (OP == OP_GRAM_NORM) return f2bf(__fdiv_rn(round_bf(v), dd));  // bf16(bf16(acc) / d^2)
    if (OP == OP_SQPOLY) return f2bf(__fadd_rn(__fmul_rn(p.b, x), __fmul_rn(p.c, v)));
    return f2bf(__fadd_rn(__fmul_rn(p.a, x), v));                   // a Y + acc
}

// The same on a pair: accumulator values v (packed fp32 pair), input word xw (two bf16);
// returns two bf16.  Rounding is identical to epi_value (each product and sum rounded).
template <int OP>
__device__ __forceinline__ uint32_t epi_pair(uint64_t v, uint32_t xw, uint64_t coef_x,
                                             uint64_t coef_v, float dd) {
    if (OP == OP_GRAM) return f2_to_bf2(v);
    if (OP == OP_GRAM_NORM) {
        // bf16(bf16(acc) / d^2), the quotient correctly rounded in fp32
        const float lo = __fdiv_rn(round_bf(__uint_as_float(static_cast<uint32_t>(v))), dd);
        const float hi = __fdiv_rn(round_bf(__uint_as_float(static_cast<uint32_t>(v >> 32))), dd);
        return f2_to_bf2(f2_pack(lo, hi));
    }
    const uint64_t t = f2_mul(coef_x, bf2_to_f2(xw));  // b A  or  a Y
    if (OP == OP_SQPOLY) return f2_to_bf2(f2_add(t, f2_mul(coef_v, v)));  // + c acc
    return f2_to_bf2(f2_add(t, v));                                          // + acc
}

template <int OP>
__global__ void __launch_bounds__(GEMM_THREADS, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    using TR = OpTraits<OP>;
    constexpr int BN = TR::BN;
    constexpr int STAGES = TR::STAGES;
    constexpr int NQ = TR::NQ;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t mma_done_bar;
    __shared__ __align__(8) uint64_t epi_bar[NQ];  // epilogue input loads, one per quarter
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int aborted;

    pdl_allow_next();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs), 1 = peer
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 2 * 4 * EPI_GROUPS);  // each epilogue warp, both CTAs
        }
        for (int q = 0; q < NQ; ++q) mbar_init(&epi_bar[q], 1);
        mbar_init(&mma_done_bar, 1);
        fence_mbar_init();
        aborted = 0;
    }
    if (threadIdx.x == 32) {
        for (int i = 0; i < p.nbanks; ++i) {
            tma_prefetch_desc(&p.bank[i].tm_a);
            tma_prefetch_desc(&p.bank[i].tm_b);
            if (TR::has_in) tma_prefetch_desc(&p.bank[i].tm_c);
            tma_prefetch_desc(&p.bank[i].tm_d);
            if (TR::has_t) tma_prefetch_desc(&p.bank[i].tm_e);
        }
    }
    if (warp == 1) tmem_alloc_pair(&tmem_slot, TR::TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    pdl_wait_previous();  // everything above overlapped the previous kernel's tail
    const uint32_t tmem = tmem_slot;
    int issued = 0;        // producer: k-blocks whose loads were armed (in the whole CTA life)
    int epi_tiles = 0;     // epilogue: tiles whose input staging loads were armed

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int it = 0;
            for (int k = 0;; ++k) {
                const int t = snake_tile(k, pair, npairs);
                if (t >= p.total_tiles || aborted) break;
                const TileCoord c = decode_tile<OP>(p, t);
                const GemmBank& bk = p.bank[c.bi];
                const int arow = c.ti * PAIR + TILE * rank;  // this CTA's A rows
                const int bofs = c.tj * PAIR + TILE * rank;  // this CTA's B rows (or Y columns)
                for (int kb = 0; kb < bk.num_kb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t r = static_cast<uint32_t>(it / STAGES);
                    if (!mbar_wait(&empty_bar[s], (r & 1u) ^ 1u, p.err)) {
                        aborted = 1;
                        break;
                    }
                    uint8_t* sa = smem + s * TR::STAGE;
                    uint8_t* sb = sa + TR::A_STAGE;
                    // both CTAs' bytes complete on the leader's barrier of this stage
                    const uint32_t fb = map_to_rank(&full_bar[s], 0);
                    if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], 2 * TR::STAGE);
                    tma_load_3d_pair(sa, &bk.tm_a, fb, kb * BK, arow, c.mat);
                    if (TR::xupdate) {
                        // Y rows kb*64 .. +63 (the contraction index), this CTA's 128 of the
                        // tile's columns in two 64-column boxes: MN-major chunks 8 KB apart.
                        tma_load_3d_pair(sb, &bk.tm_b, fb, bofs, kb * BK, c.mat);
                        tma_load_3d_pair(sb + 8192, &bk.tm_b, fb, bofs + 64, kb * BK, c.mat);
                    } else {
                        tma_load_3d_pair(sb, &bk.tm_b, fb, kb * BK, bofs, c.mat);
                    }
                    issued = it + 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (leader CTA)
            constexpr uint32_t idesc = idesc_bf16_f32(PAIR, PAIR, false, TR::xupdate);
            int it = 0;
            for (int lt = 0;; ++lt) {
                const int t = snake_tile(lt, pair, npairs);
                if (t >= p.total_tiles || aborted) break;
                const TileCoord c = decode_tile<OP>(p, t);
                const int nkb = p.bank[c.bi].num_kb;
                const int ab = lt & 1;
                const uint32_t u = static_cast<uint32_t>(lt >> 1);
                if (!mbar_wait(&tempty_bar[ab], (u & 1u) ^ 1u, p.err)) {
                    aborted = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + static_cast<uint32_t>(ab * BN);
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t r = static_cast<uint32_t>(it / STAGES);
                    if (!mbar_wait(&full_bar[s], r & 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(smem + s * TR::STAGE);
                    const uint32_t b0 = a0 + TR::A_STAGE;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a0 + kk * 32, 16, 1024);
                        const uint64_t bd = TR::xupdate ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                                                        : smem_desc_sw128(b0 + kk * 32, 16, 1024);
                        umma_bf16_pair(dacc, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    umma_commit_pair(&empty_bar[s], 3);  // frees stage s in both CTAs
                }
                if (!ok) {
                    aborted = 1;
                    break;
                }
                umma_commit_pair(&tfull_bar[ab], 3);  // accumulator ab complete in both CTAs
            }
            // every MMA has completed (in both CTAs' TMEM) once this barrier fires
            umma_commit_pair(&mma_done_bar, 3);
            mbar_wait(&mma_done_bar, 0, p.err);
        } else if (lane == 0) {
            // peer CTA: its TMEM is written by the leader's MMAs; wait for the last one
            mbar_wait(&mma_done_bar, 0, p.err);
        }
    } else {
        // ---------------- epilogue: warps 2-9, TMEM lane quadrant = warp % 4
        const int quad = warp & 3;
        const int grp = (warp - 2) >> 2;          // column half of this warp group
        const int r = quad * 32 + lane;           // row within the tile
        const bool leader = ((warp - 2) & 3) == 0 && lane == 0;
        uint8_t* stg = smem + STAGES * TR::STAGE;  // staging boxes (1024-aligned)
        const uint32_t tempty_leader0 = map_to_rank(&tempty_bar[0], 0);
        const uint32_t tempty_leader1 = map_to_rank(&tempty_bar[1], 0);
        const uint64_t coef_x = f2_pack(OP == OP_SQPOLY ? p.b : p.a, OP == OP_SQPOLY ? p.b : p.a);
        const uint64_t coef_v = f2_pack(p.c, p.c);
        for (int lt = 0;; ++lt) {
            const int t = snake_tile(lt, pair, npairs);
            if (t >= p.total_tiles || aborted) break;
            const TileCoord c = decode_tile<OP>(p, t);
            const GemmBank& bk = p.bank[c.bi];
            const int ab = lt & 1;
            const uint32_t u = static_cast<uint32_t>(lt >> 1);
            const int row0 = c.ti * PAIR + TILE * rank;  // this CTA's first output row
            const int col0 = c.tj * PAIR;                // first column
            // what this tile stores: the tile itself, and/or its transpose
            const bool to_direct = TR::sym || OP == OP_XUPDATE || (OP == OP_XUPDATE_OUT && !bk.tall);
            const bool to_mirror = (TR::sym && c.ti != c.tj) || (OP == OP_XUPDATE_OUT && bk.tall);
            const bool staged = OP != OP_XUPDATE_OUT || bk.out_tma;
            float dd = 0.f;
            if (OP == OP_GRAM_NORM) {
                const float d = bk.d[c.mat];
                dd = __fmul_rn(d, d);
            }

            const uint32_t in_phase = static_cast<uint32_t>(epi_tiles) & 1u;
            if (staged && TR::has_in) {
                // this group's quarters of the tile's input, once this group's earlier
                // stores have finished reading the boxes
                if (leader) {
                    bulk_wait_read_all();
                    for (int q = 2 * grp; q < 2 * grp + 2; ++q) {
                        mbar_arrive_expect_tx(&epi_bar[q], QBOX);
                        tma_load_3d(stg + q * QBOX, &bk.tm_c, &epi_bar[q], col0 + 64 * q, row0, c.mat);
                    }
                }
                ++epi_tiles;
            }
            if (!mbar_wait(&tfull_bar[ab], u & 1u, p.err)) {
                aborted = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(ab * BN);

            if (!staged) {
                // OP_XUPDATE_OUT into an `out` whose rows are not 16-byte aligned: plain
                // bounds-checked stores straight from the accumulator (this group's half).
                const int m = bk.m, n = bk.n;
                uint16_t* out = bk.dst + static_cast<size_t>(c.mat) * m * n;
                const int row = row0 + r;
#pragma unroll 1
                for (int cc = 4 * grp; cc < 4 * grp + 4; ++cc) {
                    const int cb = col0 + cc * 32;
                    float x[32];
                    load32_bf16(bk.src + (static_cast<size_t>(c.mat) * bk.s_pad + row) * bk.L_pad + cb, x);
                    float v[32];
                    tmem_ld_32x32b_x32(tbase + cc * 32, v);
                    uint16_t o[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] = epi_value<OP>(p, v[q], x[q], dd);
                    if (!bk.tall) {
                        if (row < m)
                            for (int q = 0; q < 32; ++q)
                                if (cb + q < n) out[static_cast<size_t>(row) * n + cb + q] = o[q];
                    } else if (row < n) {
                        for (int q = 0; q < 32; ++q)
                            if (cb + q < m) out[static_cast<size_t>(cb + q) * n + row] = o[q];
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(ab ? tempty_leader1 : tempty_leader0);
                continue;
            }

            bool ok = true;
            for (int q = 2 * grp; q < 2 * grp + 2; ++q) {
                // direct box: the tile's q-th input box (updated in place), or the group's
                // output box; transposed box: the group's
                uint8_t* dbox = stg + (TR::has_in ? q : grp) * QBOX;
                uint8_t* tbox = stg + (TR::NDIR + grp) * QBOX;  // 64 rows x 128 cols, plain
                if (!TR::has_in || TR::has_t) {
                    // the boxes written below must be free of this group's last store
                    if (leader) bulk_wait_read_all();
                    named_barrier_sync(1 + grp, 128);
                }
                if (TR::has_in && !mbar_wait(&epi_bar[q], in_phase, p.err)) {
                    ok = false;
                    break;
                }
                uint8_t* drow = dbox + r * 128;
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float v[32];
                    tmem_ld_32x32b_x32(tbase + q * 64 + cc * 32, v);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        // 16-byte chunk j of this 128-byte row sits at chunk j ^ (r % 8)
                        const int j = cc * 4 + w;
                        uint4* cp = reinterpret_cast<uint4*>(drow + ((j ^ (r & 7)) << 4));
                        uint32_t xw[4] = {0u, 0u, 0u, 0u};
                        if (TR::has_in) {
                            const uint4 x = *cp;
                            xw[0] = x.x; xw[1] = x.y; xw[2] = x.z; xw[3] = x.w;
                        }
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = epi_pair<OP>(f2_pack(v[8 * w + 2 * e], v[8 * w + 2 * e + 1]), xw[e],
                                                coef_x, coef_v, dd);
                        if (to_direct) *cp = make_uint4(o[0], o[1], o[2], o[3]);
                        if (TR::has_t && to_mirror) {
                            // transposed box: element (row r, column 8j + e) at [8j + e][r]
                            uint16_t* tcol = reinterpret_cast<uint16_t*>(tbox) + r;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                tcol[(8 * j + 2 * e) * TILE] = static_cast<uint16_t>(o[e] & 0xffffu);
                                tcol[(8 * j + 2 * e + 1) * TILE] = static_cast<uint16_t>(o[e] >> 16);
                            }
                        }
                    }
                }
                if (q == 2 * grp + 1) {
                    // accumulator ab is free once every epilogue warp of both CTAs has read it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(ab ? tempty_leader1 : tempty_leader0);
                }
                fence_proxy_async_smem();
                named_barrier_sync(1 + grp, 128);
                if (leader) {
                    if (to_direct) tma_store_3d(&bk.tm_d, dbox, col0 + 64 * q, row0, c.mat);
                    if (TR::has_t && to_mirror) tma_store_3d(&bk.tm_e, tbox, row0, col0 + 64 * q, c.mat);
                    bulk_commit_group();
                }
            }
            if (!ok) {
                aborted = 1;
                break;
            }
        }
        if (leader) {
            bulk_wait_all();  // every store of this group has completed
            if (aborted && epi_tiles > 0)  // and every staging load it armed has landed
                for (int q = 2 * grp; q < 2 * grp + 2; ++q)
                    mbar_wait(&epi_bar[q], static_cast<uint32_t>(epi_tiles - 1) & 1u, p.err);
        }
    }

    __syncthreads();
    if (aborted && warp == 0 && lane == 0 && rank == 0) {
        // Let the copies still in flight land before the pair's shared memory goes away:
        // both CTAs' loads complete on the leader's barriers, and the last load armed on
        // each stage is that stage's latest phase (the peer waits in the cluster barrier).
        for (int kb = issued - STAGES < 0 ? 0 : issued - STAGES; kb < issued; ++kb)
            mbar_wait(&full_bar[kb % STAGES], (static_cast<uint32_t>(kb) / STAGES) & 1u, p.err);
    }
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while the pair still uses its memory
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, TR::TMEM_COLS);
}

static int g_max_pairs[5][64];  // co-resident CTA pairs per op and device (0 = unknown)

template <int OP>
static cudaError_t launch_op(const GemmParams& p, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // the prologue may overlap the previous kernel's tail (see pdl_wait_previous)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = OpTraits<OP>::SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int& maxp = g_max_pairs[OP][dev & 63];
    if (maxp == 0) {
        cfg.gridDim = dim3(2 * (p.sm_count / 2), 1, 1);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel<OP>, &cfg);
        if (e) return e;
        maxp = clusters > 0 ? clusters : 1;
    }
    const int pairs = p.total_tiles < maxp ? p.total_tiles : maxp;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<OP>, p);
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

int gemm_tile_cols(GemmOp) { return PAIR; }

cudaError_t gemm_prepare() {
    cudaError_t e;
#define ANVIL_SET_SMEM(OPV)                                                                  \
    if ((e = cudaFuncSetAttribute(gemm_kernel<OPV>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  OpTraits<OPV>::SMEM)))                                     \
        return e;
    ANVIL_SET_SMEM(OP_GRAM)
    ANVIL_SET_SMEM(OP_GRAM_NORM)
    ANVIL_SET_SMEM(OP_SQPOLY)
    ANVIL_SET_SMEM(OP_XUPDATE)
    ANVIL_SET_SMEM(OP_XUPDATE_OUT)
#undef ANVIL_SET_SMEM
    return cudaSuccess;
}

}  // namespace anvil
