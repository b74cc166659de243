// anvil_api.cu -- libanvil's C ABI (include/anvil.h): argument checks, the call-wide
// workspace layout, TMA tensor maps, and the launch sequence of one ANVIL step
// (page "modded-nanogpt track_1_short/optim/anvil.py", anvil_cascade):
//
//   momentum + cast (+ diagonal partials)   -> Y0 = X_raw          (momentum_kernel)
//   d = sqrt(tr) * margin + eps             (tr from the bf16 diagonal of the first Gram;
//                                             norm_d_kernel, which also zeroes the
//                                             cascade's completion counters)
//   the cascade (cascade_kernel, one persistent launch over every phase):
//     A = bf16(bf16(Y0 Y0^T) / d^2);  Y1 = bf16(Y0 / d)
//     map k = 0..nmaps-1, reading Y[(k+1)%2], writing Y[k%2] (out for the last map):
//       [k > 0] A = bf16(Y Y^T);  B = bf16(b A + c A A);  Y' = bf16(a Y + B Y)
//
// Three launches per step for any number of banks; a traced step runs the cascade one
// phase per launch and copies the intermediate values out between them.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>


#include "../../include/anvil.h"
#include "anvil_internal.h"
#include "anvil_adam.h"
#include "anvil_schedule.h"
#include "anvil_tail.h"

using namespace anvil;

static_assert(ANVIL_MAX_MAPS <= MAX_CASCADE_MAPS, "phase table too small for ANVIL_MAX_MAPS");
static_assert(TL_ITEMS == ANVIL_TIMELINE_ITEMS && TL_FIELDS == 16, "timeline layout of include/anvil.h");
static_assert(sizeof(CascadeParams) <= 32764, "cascade parameters exceed the kernel parameter limit");

namespace {

thread_local char g_last_error[256] = "";

anvil_status cuda_fail(cudaError_t e, const char* where) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
    return ANVIL_ERR_CUDA;
}

// ANVIL_MAPS as printed on the page (the ANVIL section of anvil.py, record #360).
const anvil_map kAnvilMaps[6] = {
    {3.923798038567f, -6.095026865488f, 3.905234618423f},
    {3.278126713798f, -3.328923386476f, 0.989127286973f},
    {3.505298394150f, -5.137358782410f, 1.968325560615f},
    {2.815058591845f, -3.685181239622f, 1.417196497642f},
    {2.245503932403f, -2.443826979899f, 0.963091710461f},
    {2.256537145403f, -2.166840097229f, 0.929501253245f},
};

// ---------------------------------------------------------------- per-device set-up
struct DeviceState {
    bool ready = false;
    unsigned* err = nullptr;
    int sm_count = 0;
};
std::mutex g_dev_mutex;
DeviceState g_dev[64];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Checks the device is sm_103, sets kernel attributes, finds the error word and the
// tensor-map encoder.  Once per device; no allocation, no synchronisation.
anvil_status device_setup(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return ANVIL_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3) {
            snprintf(g_last_error, sizeof(g_last_error),
                     "device %d is sm_%d%d; libanvil is built for sm_103a only", dev, major, minor);
            return ANVIL_ERR_DEVICE;
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return cuda_fail(e == cudaSuccess ? cudaErrorSymbolNotFound : e,
                                 "cuTensorMapEncodeTiled lookup");
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        if ((e = gemm_prepare())) return cuda_fail(e, "cudaFuncSetAttribute");
        if ((e = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        st.err = device_error_word();
        if (!st.err) return cuda_fail(cudaGetLastError(), "cudaGetSymbolAddress(error word)");
        st.ready = true;
    }
    *out = &st;
    return ANVIL_OK;
}

// ---------------------------------------------------------------- launch profiling
struct Profiler {
    std::mutex mu;
    bool active = false;
    int cap = 0, used = 0;
    cudaEvent_t* ev = nullptr;  // 2 * cap events
    int* kind = nullptr;
};
Profiler g_prof;

// Runs `launch`, bracketed by two events on `stream` when profiling is on.  A timed
// launch holds the profiler's lock throughout, so anvil_profile_end on another thread
// cannot destroy its events in between.
template <class F>
cudaError_t profiled(int kind, cudaStream_t stream, F&& launch) {
    std::unique_lock<std::mutex> lock(g_prof.mu);
    if (!g_prof.active || g_prof.used >= g_prof.cap) {
        lock.unlock();
        return launch();
    }
    const int slot = g_prof.used++;
    g_prof.kind[slot] = kind;
    cudaError_t e;
    if ((e = cudaEventRecord(g_prof.ev[2 * slot], stream))) return e;
    if ((e = launch())) return e;
    return cudaEventRecord(g_prof.ev[2 * slot + 1], stream);
}

// ---------------------------------------------------------------- geometry and layout
struct Geom {
    int g, m, n, tall, s, L, s_pad, L_pad, nlb, mat_begin;
    size_t part_off, y_off, a_off;  // element offsets into the call-wide arrays
};

struct Layout {
    Geom bank[ANVIL_MAX_BANKS];
    int nbanks, total_mats;
    size_t part_elems, y_elems, a_elems;
    size_t off_d, off_cnt, off_part, off_y0, off_y1, off_a, off_b, total;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// The cascade kernel's bank order: the call's banks, heaviest tiles first (they open
// every phase), ties in call order.
void cascade_bank_order(const Geom* bank, int nbanks, int* order) {
    for (int i = 0; i < nbanks; ++i) order[i] = i;
    std::stable_sort(order, order + nbanks, [&](int x, int y) {
        const long long wx = static_cast<long long>(bank[x].s_pad) * bank[x].L_pad;
        const long long wy = static_cast<long long>(bank[y].s_pad) * bank[y].L_pad;
        return wx > wy;
    });
}

anvil_status make_layout(const anvil_bank_desc* banks, int nbanks, Layout* L) {
    if (!banks || nbanks < 1 || nbanks > ANVIL_MAX_BANKS) return ANVIL_ERR_INVALID_ARG;
    L->nbanks = nbanks;
    L->total_mats = 0;
    L->part_elems = L->y_elems = L->a_elems = 0;
    for (int i = 0; i < nbanks; ++i) {
        const anvil_bank_desc& b = banks[i];
        if (b.g < 1 || b.m < 1 || b.n < 1) return ANVIL_ERR_INVALID_ARG;
        if (b.m > ANVIL_MAX_DIM || b.n > ANVIL_MAX_DIM || b.g > ANVIL_MAX_BATCH)
            return ANVIL_ERR_UNSUPPORTED_SHAPE;
        Geom& G = L->bank[i];
        G.g = b.g;
        G.m = b.m;
        G.n = b.n;
        G.tall = b.m > b.n;
        G.s = G.tall ? b.n : b.m;
        G.L = G.tall ? b.m : b.n;
        G.s_pad = round_up(G.s, PAIR);
        G.L_pad = round_up(G.L, LPAD);
        G.nlb = G.L_pad / LBLK;
        G.mat_begin = L->total_mats;
        L->total_mats += b.g;
        G.part_off = L->part_elems;
        G.y_off = L->y_elems;
        G.a_off = L->a_elems;
        L->part_elems += static_cast<size_t>(b.g) * G.nlb * G.s_pad;
        L->y_elems += static_cast<size_t>(b.g) * G.s_pad * G.L_pad;
        L->a_elems += static_cast<size_t>(b.g) * G.s_pad * G.s_pad;
    }
    // 32-bit tile and item counts (the momentum grid, the cascade's item numbers: at most
    // MAX_PHASES items per 256 x 256 block of Y) hold below 2^40 elements of Y, 2 TB
    if (L->y_elems > (static_cast<size_t>(1) << 40)) return ANVIL_ERR_UNSUPPORTED_SHAPE;
    L->off_d = 0;
    L->off_cnt = align256(L->off_d + sizeof(float) * L->total_mats);
    L->off_part = align256(L->off_cnt + sizeof(unsigned) * (L->total_mats + SCHED_COUNTERS));
    L->off_y0 = align256(L->off_part + sizeof(float) * L->part_elems);
    L->off_y1 = align256(L->off_y0 + 2 * L->y_elems);
    L->off_a = align256(L->off_y1 + 2 * L->y_elems);
    L->off_b = align256(L->off_a + 2 * L->a_elems);
    L->total = align256(L->off_b + 2 * L->a_elems);
    return ANVIL_OK;
}

struct Range {
    uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

anvil_status check_banks(const anvil_bank_desc* banks, int nbanks) {
    Range rg[ANVIL_MAX_BANKS][4];
    for (int i = 0; i < nbanks; ++i) {
        const anvil_bank_desc& b = banks[i];
        if (!b.grad || !b.velocity || !b.out) return ANVIL_ERR_INVALID_ARG;
        const uintptr_t gsz = b.grad_bf16 ? 2 : 4;
        if ((reinterpret_cast<uintptr_t>(b.grad) & (gsz - 1)) || (reinterpret_cast<uintptr_t>(b.velocity) & 3) ||
            (reinterpret_cast<uintptr_t>(b.out) & 1) || (reinterpret_cast<uintptr_t>(b.tail_link) & 255))
            return ANVIL_ERR_ALIGNMENT;
        const size_t cnt = static_cast<size_t>(b.g) * b.m * b.n;
        rg[i][0] = {reinterpret_cast<uintptr_t>(b.grad), reinterpret_cast<uintptr_t>(b.grad) + gsz * cnt};
        rg[i][1] = {reinterpret_cast<uintptr_t>(b.velocity), reinterpret_cast<uintptr_t>(b.velocity + 2 * cnt)};
        rg[i][2] = {reinterpret_cast<uintptr_t>(b.out), reinterpret_cast<uintptr_t>(b.out + cnt)};
        const uintptr_t lk = reinterpret_cast<uintptr_t>(b.tail_link);
        rg[i][3] = {lk, lk ? lk + link_layout(b.g, b.m, b.n).total : lk};
    }
    // written buffers (velocity, out, tail_link) must overlap nothing else of the call
    for (int i = 0; i < nbanks; ++i)
        for (int w = 1; w <= 3; ++w)
            for (int j = 0; j < nbanks; ++j)
                for (int k = 0; k < 4; ++k) {
                    if (i == j && k == w) continue;
                    if (overlap(rg[i][w], rg[j][k])) return ANVIL_ERR_ALIAS;
                }
    return ANVIL_OK;
}

anvil_status check_maps(const anvil_map* maps, int nmaps) {
    if (!maps || nmaps < 1 || nmaps > ANVIL_MAX_MAPS) return ANVIL_ERR_INVALID_ARG;
    return ANVIL_OK;
}

// 3-D bf16 tensor map over [g][rows][cols], box {box0, box1, 1}, 128-byte swizzle or none.
anvil_status encode_map(CUtensorMap* map, void* base, int g, int rows, int cols, int box0, int box1,
                        bool swizzle = true) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(g)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                                   static_cast<cuuint64_t>(rows) * cols * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(box0), static_cast<cuuint32_t>(box1), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (%d)",
                 static_cast<int>(r));
        return ANVIL_ERR_CUDA;
    }
    return ANVIL_OK;
}

// Device pointers of one bank's slices of the workspace.
struct BankPtrs {
    uint16_t* y[2];
    uint16_t* a;
    uint16_t* b;
    float* part;
    float* d;
    CUtensorMap tm[TM_COUNT];
    bool out_tma;
};

anvil_status run_step(const anvil_bank_desc* banks, int nbanks, const anvil_scalars* d_scalars,
                      const anvil_map* maps, int nmaps, float margin, float eps, void* workspace,
                      size_t ws_bytes, cudaStream_t stream, const anvil_trace* trace) {
    // Every argument check comes before any CUDA call.
    anvil_status st;
    Layout L;
    if ((st = make_layout(banks, nbanks, &L)) != ANVIL_OK) return st;
    if ((st = check_banks(banks, nbanks)) != ANVIL_OK) return st;
    if ((st = check_maps(maps, nmaps)) != ANVIL_OK) return st;
    if (!workspace || ws_bytes < L.total) return ANVIL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return ANVIL_ERR_ALIGNMENT;
    {
        const Range wr = {reinterpret_cast<uintptr_t>(workspace),
                          reinterpret_cast<uintptr_t>(workspace) + L.total};
        for (int i = 0; i < nbanks; ++i) {
            const size_t cnt = static_cast<size_t>(banks[i].g) * banks[i].m * banks[i].n;
            const uintptr_t gsz = banks[i].grad_bf16 ? 2 : 4;
            const uintptr_t lk = reinterpret_cast<uintptr_t>(banks[i].tail_link);
            const Range r[4] = {{reinterpret_cast<uintptr_t>(banks[i].grad), reinterpret_cast<uintptr_t>(banks[i].grad) + gsz * cnt},
                                {reinterpret_cast<uintptr_t>(banks[i].velocity), reinterpret_cast<uintptr_t>(banks[i].velocity + 2 * cnt)},
                                {reinterpret_cast<uintptr_t>(banks[i].out), reinterpret_cast<uintptr_t>(banks[i].out + cnt)},
                                {lk, lk ? lk + link_layout(banks[i].g, banks[i].m, banks[i].n).total : lk}};
            for (int k = 0; k < 4; ++k)
                if (overlap(wr, r[k])) return ANVIL_ERR_ALIAS;
        }
    }
    if (d_scalars && (reinterpret_cast<uintptr_t>(d_scalars) & 3)) return ANVIL_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    if ((st = device_setup(&dev)) != ANVIL_OK) return st;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* d_all = reinterpret_cast<float*>(ws + L.off_d);
    BankPtrs P[ANVIL_MAX_BANKS];
    for (int i = 0; i < nbanks; ++i) {
        const Geom& G = L.bank[i];
        BankPtrs& B = P[i];
        B.y[0] = reinterpret_cast<uint16_t*>(ws + L.off_y0) + G.y_off;
        B.y[1] = reinterpret_cast<uint16_t*>(ws + L.off_y1) + G.y_off;
        B.a = reinterpret_cast<uint16_t*>(ws + L.off_a) + G.a_off;
        B.b = reinterpret_cast<uint16_t*>(ws + L.off_b) + G.a_off;
        B.part = reinterpret_cast<float*>(ws + L.off_part) + G.part_off;
        B.d = d_all + G.mat_begin;
        for (int k = 0; k < 2; ++k) {
            if ((st = encode_map(&B.tm[TM_YK0 + k], B.y[k], G.g, G.s_pad, G.L_pad, BK, TILE))) return st;
            if ((st = encode_map(&B.tm[TM_YN0 + k], B.y[k], G.g, G.s_pad, G.L_pad, BK, BK))) return st;
        }
        if ((st = encode_map(&B.tm[TM_A], B.a, G.g, G.s_pad, G.s_pad, BK, TILE))) return st;
        if ((st = encode_map(&B.tm[TM_B], B.b, G.g, G.s_pad, G.s_pad, BK, TILE))) return st;
        if ((st = encode_map(&B.tm[TM_AN], B.a, G.g, G.s_pad, G.s_pad, BK, BK))) return st;
        if ((st = encode_map(&B.tm[TM_BN], B.b, G.g, G.s_pad, G.s_pad, BK, BK))) return st;
        // the last X-update stores `out` [g, m, n] by TMA when its rows are 16-byte aligned:
        // boxes of Y (64 columns x 128 rows) for a wide bank, transposed 64 x 64 boxes for a
        // tall one (out = Y^T); other shapes take plain stores
        memset(&B.tm[TM_OUT], 0, sizeof(CUtensorMap));
        B.out_tma = (G.n % 8 == 0) && !(reinterpret_cast<uintptr_t>(banks[i].out) & 15);
        if (B.out_tma &&
            (st = encode_map(&B.tm[TM_OUT], banks[i].out, G.g, G.m, G.n, BK, G.tall ? BK : TILE)))
            return st;
    }

    cudaError_t e;
    // ---- momentum + cast + diagonal partials
    {
        MomentumParams mp;
        memset(&mp, 0, sizeof(mp));
        mp.nbanks = nbanks;
        mp.dev_scalars = reinterpret_cast<const float*>(d_scalars);
        mp.err = dev->err;
        int tiles = 0;
        for (int i = 0; i < nbanks; ++i) {
            const Geom& G = L.bank[i];
            const anvil_bank_desc& b = banks[i];
            MomentumBank& M = mp.bank[i];
            M.grad = b.grad;
            M.velocity = b.velocity;
            M.y = P[i].y[0];
            M.part = P[i].part;
            M.g = G.g;
            M.m = G.m;
            M.n = G.n;
            M.tall = G.tall;
            M.s_pad = G.s_pad;
            M.L_pad = G.L_pad;
            M.nlb = G.nlb;
            M.tiles_r = (G.tall ? G.L_pad : G.s_pad) / LBLK;
            M.tiles_c = (G.tall ? G.s_pad : G.L_pad) / LBLK;
            M.tile_begin = tiles;
            M.grad_bf16 = b.grad_bf16 ? 1 : 0;
            M.vec4 = (G.n % 4 == 0) && !(reinterpret_cast<uintptr_t>(b.grad) & (b.grad_bf16 ? 7 : 15)) &&
                     !(reinterpret_cast<uintptr_t>(b.velocity) & 15);
            if (b.tail_link) {
                const LinkLayout lk = link_layout(G.g, G.m, G.n);
                M.gate = static_cast<uint64_t*>(b.tail_link);
                M.nck = lk.nck;
            }
            M.momentum = b.scalars.momentum;
            M.fast_beta = b.scalars.fast_beta;
            M.fast_weight = b.scalars.fast_weight;
            M.slow_beta = b.scalars.slow_beta;
            tiles += G.g * M.tiles_r * M.tiles_c;
        }
        mp.total_tiles = tiles;
        if ((e = profiled(ANVIL_KERNEL_MOMENTUM, stream, [&] { return launch_momentum(mp, stream); })))
            return cuda_fail(e, "momentum launch");
    }
    // ---- d
    NormParams np;
    memset(&np, 0, sizeof(np));
    np.nbanks = nbanks;
    np.total_mats = L.total_mats;
    np.margin = margin;
    np.eps = eps;
    np.d = d_all;
    np.counters = reinterpret_cast<unsigned*>(ws + L.off_cnt);
    np.err = dev->err;
    for (int i = 0; i < nbanks; ++i) {
        const Geom& G = L.bank[i];
        NormBank& N = np.bank[i];
        N.part = P[i].part;
        N.g = G.g;
        N.s_pad = G.s_pad;
        N.L_pad = G.L_pad;
        N.nlb = G.nlb;
        N.mat_begin = G.mat_begin;
    }
    if ((e = profiled(ANVIL_KERNEL_NORM_D, stream, [&] { return launch_norm_d(np, stream); })))
        return cuda_fail(e, "norm_d launch");
    if (trace) {
        const Geom& G = L.bank[0];
        if (trace->X_raw && (e = launch_extract_x(P[0].y[0], trace->X_raw, G.g, G.m, G.n, G.tall,
                                                  G.s_pad, G.L_pad, stream)))
            return cuda_fail(e, "trace");
        if (trace->d && (e = cudaMemcpyAsync(trace->d, P[0].d, sizeof(float) * G.g,
                                             cudaMemcpyDeviceToDevice, stream)))
            return cuda_fail(e, "trace");
    }
    // ---- X / d
    NormXParams xp;
    memset(&xp, 0, sizeof(xp));
    xp.nbanks = nbanks;
    for (int i = 0; i < nbanks; ++i) {
        const Geom& G = L.bank[i];
        NormXBank& X = xp.bank[i];
        X.y0 = P[i].y[0];
        X.y1 = P[i].y[1];
        X.d = P[i].d;
        // s_pad is a multiple of PAIR and L_pad of LPAD: a matrix is a whole number of blocks
        X.blocks_per_mat = static_cast<int>(static_cast<long long>(G.s_pad) * G.L_pad / 8 / NX_BLOCK_CHUNKS);
        X.block_begin = xp.total_blocks;
        xp.total_blocks += G.g * X.blocks_per_mat;
    }
    if ((e = profiled(ANVIL_KERNEL_NORMALIZE, stream, [&] { return launch_normalize(xp, stream); })))
        return cuda_fail(e, "normalize launch");
    if (trace && trace->X) {
        const Geom& G = L.bank[0];
        if ((e = launch_extract_x(P[0].y[1], trace->X, G.g, G.m, G.n, G.tall, G.s_pad, G.L_pad, stream)))
            return cuda_fail(e, "trace");
    }

    // ---- the cascade: every phase of every map in one persistent launch (one launch per
    // phase when tracing, with the intermediate values copied out between them)
    CascadeParams cparams;
    CascadeParams* cp = &cparams;
    memset(cp, 0, sizeof(*cp));
    cp->nbanks = nbanks;
    cp->sm_count = dev->sm_count;
    cp->chain = reinterpret_cast<unsigned*>(ws + L.off_cnt);
    unsigned* sched_ctr = cp->chain + L.total_mats;  // [SCHED_COUNTERS]
    cp->err = dev->err;
    int order[ANVIL_MAX_BANKS];
    cascade_bank_order(L.bank, nbanks, order);
    for (int q = 0; q < nbanks; ++q) {
        const int i = order[q];
        const Geom& G = L.bank[i];
        const BankPtrs& B = P[i];
        CascadeBank& cb = cp->bank[q];
        memcpy(cb.tm, B.tm, sizeof(cb.tm));
        cb.a = B.a;
        cb.b = B.b;
        cb.out = banks[i].out;
        cb.y0 = B.y[0];
        cb.y1 = B.y[1];
        cb.d = B.d;
        cb.g = G.g;
        cb.s_pad = G.s_pad;
        cb.L_pad = G.L_pad;
        cb.m = G.m;
        cb.n = G.n;
        cb.tall = G.tall;
        cb.out_tma = B.out_tma ? 1 : 0;
        cb.T = G.s_pad / PAIR;
        cb.ntl = G.L_pad / PAIR;
        cb.mat_begin = G.mat_begin;
    }
    build_phases(cp, maps, nmaps);
    int phase_run[MAX_PHASES + 1];
    order_phase_major(cp, phase_run);
    auto run_range = [&](int first, int end, int kind, int slot) -> anvil_status {
        cp->first_run = first;
        cp->end_run = end;
        cp->next_item = sched_ctr + slot;
        cudaError_t ee = profiled(kind, stream, [&] { return launch_cascade(*cp, stream); });
        return ee ? cuda_fail(ee, "cascade launch") : ANVIL_OK;
    };
    if (!trace) return run_range(0, cp->nruns, ANVIL_KERNEL_CASCADE, 0);

    static const int kinds[5] = {ANVIL_KERNEL_GRAM, ANVIL_KERNEL_GRAM_NORM, ANVIL_KERNEL_SQPOLY,
                                 ANVIL_KERNEL_XUPDATE, ANVIL_KERNEL_XUPDATE_OUT};
    const Geom& G0 = L.bank[0];
    const size_t nx1 = static_cast<size_t>(G0.g) * G0.m * G0.n;
    const size_t na1 = static_cast<size_t>(G0.g) * G0.s * G0.s;
    for (int ph = 0, k = 0; ph < cp->nphases; ++ph) {
        const int op = cp->phase[ph].op;
        if ((st = run_range(phase_run[ph], phase_run[ph + 1], kinds[op], 1 + ph))) return st;
        if ((op == OP_GRAM || op == OP_GRAM_NORM) && trace->A &&
            (e = launch_extract_sq(P[0].a, trace->A + k * na1, G0.g, G0.s, G0.s_pad, stream)))
            return cuda_fail(e, "trace");
        if (op == OP_SQPOLY && trace->B &&
            (e = launch_extract_sq(P[0].b, trace->B + k * na1, G0.g, G0.s, G0.s_pad, stream)))
            return cuda_fail(e, "trace");
        if (op == OP_XUPDATE || op == OP_XUPDATE_OUT) {
            if (trace->X) {
                if (op == OP_XUPDATE_OUT) {
                    if ((e = cudaMemcpyAsync(trace->X + (k + 1) * nx1, banks[0].out, 2 * nx1,
                                             cudaMemcpyDeviceToDevice, stream)))
                        return cuda_fail(e, "trace");
                } else if ((e = launch_extract_x(P[0].y[k & 1], trace->X + (k + 1) * nx1, G0.g, G0.m,
                                                 G0.n, G0.tall, G0.s_pad, G0.L_pad, stream))) {
                    return cuda_fail(e, "trace");
                }
            }
            ++k;
        }
    }
    return ANVIL_OK;
}

// Workspace bytes of one call after run_step's checks that need no workspace or device
// (shapes, pointers, maps); 0 with *st set when one fails.
size_t checked_layout_bytes(const anvil_bank_desc* bank, const anvil_map* maps, int nmaps,
                            anvil_status* st) {
    Layout L;
    if ((*st = make_layout(bank, 1, &L)) != ANVIL_OK) return 0;
    if ((*st = check_banks(bank, 1)) != ANVIL_OK) return 0;
    if ((*st = check_maps(maps, nmaps)) != ANVIL_OK) return 0;
    return L.total;
}

// ---------------------------------------------------------------- update tail
struct TailLayout {
    int total_mats;
    size_t lanes_total;  // sum over banks of g * nl
    size_t off_power, off_scale, total;
    size_t lane_off[ANVIL_MAX_BANKS];
};

anvil_status make_tail_layout(const anvil_tail_desc* banks, int nbanks, TailLayout* T) {
    if (!banks || nbanks < 1 || nbanks > ANVIL_MAX_BANKS) return ANVIL_ERR_INVALID_ARG;
    T->total_mats = 0;
    T->lanes_total = 0;
    for (int i = 0; i < nbanks; ++i) {
        const anvil_tail_desc& b = banks[i];
        if (b.g < 1 || b.m < 1 || b.n < 1) return ANVIL_ERR_INVALID_ARG;
        if (b.m > ANVIL_MAX_DIM || b.n > ANVIL_MAX_DIM || b.g > ANVIL_MAX_BATCH)
            return ANVIL_ERR_UNSUPPORTED_SHAPE;
        T->lane_off[i] = T->lanes_total;
        T->lanes_total += static_cast<size_t>(b.g) * (b.m >= b.n ? b.m : b.n);
        T->total_mats += b.g;
    }
    T->off_power = 0;
    T->off_scale = align256(sizeof(float) * T->lanes_total);
    T->total = align256(T->off_scale + sizeof(float) * T->lanes_total);
    return ANVIL_OK;
}

anvil_status check_tail(const anvil_tail_desc* banks, int nbanks) {
    Range rg[ANVIL_MAX_BANKS][7];
    for (int i = 0; i < nbanks; ++i) {
        const anvil_tail_desc& b = banks[i];
        if (!b.update || !b.velocity || !b.lane_energy || !b.param || !b.mantissa || !b.eff_lr)
            return ANVIL_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(b.update) & 1) || (reinterpret_cast<uintptr_t>(b.param) & 1) ||
            (reinterpret_cast<uintptr_t>(b.mantissa) & 1) || (reinterpret_cast<uintptr_t>(b.velocity) & 3) ||
            (reinterpret_cast<uintptr_t>(b.lane_energy) & 3) || (reinterpret_cast<uintptr_t>(b.eff_lr) & 3) ||
            (reinterpret_cast<uintptr_t>(b.tail_link) & 255))
            return ANVIL_ERR_ALIGNMENT;
        const size_t cnt = static_cast<size_t>(b.g) * b.m * b.n;
        const size_t nl = static_cast<size_t>(b.g) * (b.m >= b.n ? b.m : b.n);
        rg[i][0] = {reinterpret_cast<uintptr_t>(b.lane_energy), reinterpret_cast<uintptr_t>(b.lane_energy + nl)};
        rg[i][1] = {reinterpret_cast<uintptr_t>(b.param), reinterpret_cast<uintptr_t>(b.param + cnt)};
        rg[i][2] = {reinterpret_cast<uintptr_t>(b.mantissa), reinterpret_cast<uintptr_t>(b.mantissa + cnt)};
        rg[i][3] = {reinterpret_cast<uintptr_t>(b.update), reinterpret_cast<uintptr_t>(b.update + cnt)};
        rg[i][4] = {reinterpret_cast<uintptr_t>(b.velocity), reinterpret_cast<uintptr_t>(b.velocity + 2 * cnt)};
        rg[i][5] = {reinterpret_cast<uintptr_t>(b.eff_lr), reinterpret_cast<uintptr_t>(b.eff_lr + b.g)};
        const uintptr_t lk = reinterpret_cast<uintptr_t>(b.tail_link);
        rg[i][6] = {lk, lk ? lk + link_layout(b.g, b.m, b.n).total : lk};
    }
    // written buffers (lane_energy, param, mantissa) overlap nothing else of the call
    for (int i = 0; i < nbanks; ++i)
        for (int w = 0; w < 3; ++w)
            for (int j = 0; j < nbanks; ++j)
                for (int k = 0; k < 7; ++k) {
                    if (i == j && k == w) continue;
                    if (overlap(rg[i][w], rg[j][k])) return ANVIL_ERR_ALIAS;
                }
    return ANVIL_OK;
}

// ---------------------------------------------------------------- library-owned workspace
struct OwnedWorkspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
OwnedWorkspace g_ws[64];

}  // namespace

// ---------------------------------------------------------------- fixed-scratch variant
// Scratch of anvil_bank_step_noalloc: one array per GPU, created when this library's
// device code is loaded onto that GPU and held until the process exits.  Host code may
// only use its name with cudaGetSymbolAddress; the device address differs per GPU.
static __device__ __align__(256) unsigned char g_static_scratch[ANVIL_STATIC_SCRATCH_BYTES];

namespace {
std::mutex g_static_mutex;
void* g_static_addr[64] = {nullptr};
}  // namespace

extern "C" {

int anvil_default_maps(anvil_map* maps, int cap) {
    if (maps && cap >= 6) memcpy(maps, kAnvilMaps, sizeof(kAnvilMaps));
    return 6;
}

size_t anvil_workspace_bytes(const anvil_bank_desc* banks, int nbanks) {
    Layout L;
    if (make_layout(banks, nbanks, &L) != ANVIL_OK) return 0;
    return L.total;
}

anvil_status anvil_multi_bank_step(const anvil_bank_desc* banks, int nbanks,
                                   const anvil_scalars* d_scalars, const anvil_map* maps,
                                   int nmaps, float margin, float eps, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    return run_step(banks, nbanks, d_scalars, maps, nmaps, margin, eps, workspace,
                    workspace_bytes, static_cast<cudaStream_t>(stream), nullptr);
}

size_t anvil_tail_link_bytes(int g, int m, int n) {
    if (g < 1 || m < 1 || n < 1 || g > ANVIL_MAX_BATCH || m > ANVIL_MAX_DIM || n > ANVIL_MAX_DIM) return 0;
    return link_layout(g, m, n).total;
}

size_t anvil_tail_workspace_bytes(const anvil_tail_desc* banks, int nbanks) {
    TailLayout T;
    if (make_tail_layout(banks, nbanks, &T) != ANVIL_OK) return 0;
    return T.total;
}

anvil_status anvil_update_tail(const anvil_tail_desc* banks, int nbanks, void* workspace,
                               size_t workspace_bytes, void* stream) {
    anvil_status st;
    TailLayout T;
    if ((st = make_tail_layout(banks, nbanks, &T)) != ANVIL_OK) return st;
    if ((st = check_tail(banks, nbanks)) != ANVIL_OK) return st;
    if (!workspace || workspace_bytes < T.total) return ANVIL_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return ANVIL_ERR_ALIGNMENT;
    DeviceState* dev = nullptr;
    if ((st = device_setup(&dev)) != ANVIL_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    TailParams tp;
    memset(&tp, 0, sizeof(tp));
    tp.nbanks = nbanks;
    tp.total_mats = T.total_mats;
    long long chunks = 0, rows = 0;
    int mats = 0;
    for (int i = 0; i < nbanks; ++i) {
        const anvil_tail_desc& b = banks[i];
        TailBank& B = tp.bank[i];
        B.row_begin = rows;
        rows += static_cast<long long>(b.g) * b.m;
        B.update = b.update;
        B.velocity = b.velocity;
        B.lane_energy = b.lane_energy;
        B.param = b.param;
        B.mantissa = b.mantissa;
        B.eff_lr = b.eff_lr;
        B.eff_wd = b.eff_wd;
        B.beta2 = b.beta2;
        B.g = b.g;
        B.m = b.m;
        B.n = b.n;
        B.mat_begin = mats;
        B.chunk_begin = chunks;
        B.vec8 = (b.n % 8 == 0) && !(reinterpret_cast<uintptr_t>(b.update) & 15) &&
                 !(reinterpret_cast<uintptr_t>(b.param) & 15) && !(reinterpret_cast<uintptr_t>(b.mantissa) & 15) &&
                 !(reinterpret_cast<uintptr_t>(b.velocity) & 15);
        B.power = reinterpret_cast<float*>(ws + T.off_power) + T.lane_off[i];
        B.scale = reinterpret_cast<float*>(ws + T.off_scale) + T.lane_off[i];
        if (b.tail_link) {  // the step's slow-rail sign words
            B.sign = static_cast<const uint64_t*>(b.tail_link);
            B.nck = link_layout(b.g, b.m, b.n).nck;
        }
        mats += b.g;
        chunks += static_cast<long long>(b.g) * b.m * ((b.n + 7) / 8);
    }
    tp.total_chunks = chunks;
    tp.total_rows = rows;
    cudaError_t e;
    if ((e = profiled(ANVIL_KERNEL_TAIL_POWER, s, [&] { return launch_tail_power(tp, s); })))
        return cuda_fail(e, "tail lane-power launch");
    if ((e = profiled(ANVIL_KERNEL_TAIL_SCALE, s, [&] { return launch_tail_scale(tp, s); })))
        return cuda_fail(e, "tail lane-scale launch");
    if ((e = profiled(ANVIL_KERNEL_TAIL_APPLY, s, [&] { return launch_tail_apply(tp, s); })))
        return cuda_fail(e, "tail apply launch");
    return ANVIL_OK;
}

anvil_status anvil_adam_step(float* param, const float* grad, float* exp_avg, float* exp_avg_sq,
                             size_t count, float beta1, float beta2, float eps, float step_size,
                             float eff_wd, void* stream) {
    if (!param || !grad || !exp_avg || !exp_avg_sq || count == 0) return ANVIL_ERR_INVALID_ARG;
    const uintptr_t ptrs[4] = {reinterpret_cast<uintptr_t>(param), reinterpret_cast<uintptr_t>(grad),
                               reinterpret_cast<uintptr_t>(exp_avg), reinterpret_cast<uintptr_t>(exp_avg_sq)};
    bool vec = true;
    for (int i = 0; i < 4; ++i) {
        if (ptrs[i] & 3) return ANVIL_ERR_ALIGNMENT;
        vec = vec && !(ptrs[i] & 15);
    }
    for (int i = 0; i < 4; ++i)
        for (int j = 0; j < 4; ++j)
            if (i != j && (i != 1) && overlap({ptrs[i], ptrs[i] + 4 * count}, {ptrs[j], ptrs[j] + 4 * count}))
                return ANVIL_ERR_ALIAS;
    anvil_status st;
    DeviceState* dev = nullptr;
    if ((st = device_setup(&dev)) != ANVIL_OK) return st;
    AdamParams a;
    a.p = param;
    a.g = grad;
    a.m = exp_avg;
    a.v = exp_avg_sq;
    a.count = static_cast<long long>(count);
    a.vec = vec ? 1 : 0;
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.c1 = 1.0f - beta1;
    a.c2 = 1.0f - beta2;
    a.eps = eps;
    a.step_size = step_size;
    a.eff_wd = eff_wd;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = profiled(ANVIL_KERNEL_ADAM, s, [&] { return launch_adam(a, s); });
    return e ? cuda_fail(e, "adam launch") : ANVIL_OK;
}

anvil_status anvil_bank_step_traced(const anvil_bank_desc* bank, const anvil_scalars* d_scalars,
                                    const anvil_map* maps, int nmaps, float margin, float eps,
                                    void* workspace, size_t workspace_bytes,
                                    const anvil_trace* trace, void* stream) {
    if (!trace) return ANVIL_ERR_INVALID_ARG;
    return run_step(bank, 1, d_scalars, maps, nmaps, margin, eps, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), trace);
}

anvil_status anvil_bank_step(const float* grad, float* velocity, int g, int m, int n,
                             float momentum, float fast_beta, float fast_weight, float slow_beta,
                             const anvil_map* maps, int nmaps, float margin, float eps,
                             uint16_t* out, void* stream) {
    anvil_bank_desc b;
    b.grad = grad;
    b.velocity = velocity;
    b.out = out;
    b.g = g;
    b.m = m;
    b.n = n;
    b.scalars.momentum = momentum;
    b.scalars.fast_beta = fast_beta;
    b.scalars.fast_weight = fast_weight;
    b.scalars.slow_beta = slow_beta;
    b.grad_bf16 = 0;
    b.tail_link = nullptr;
    if (!maps) {
        maps = kAnvilMaps;
        nmaps = 6;
    }
    // the argument checks and the device check come before the workspace is touched, so a
    // bad call returns the same status as anvil_multi_bank_step and allocates nothing
    anvil_status st;
    const size_t need = checked_layout_bytes(&b, maps, nmaps, &st);
    if (st != ANVIL_OK) return st;
    DeviceState* ds = nullptr;
    if ((st = device_setup(&ds)) != ANVIL_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return ANVIL_ERR_DEVICE;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        OwnedWorkspace& w = g_ws[dev];
        if (w.bytes < need) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if ((e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs)))
                return cuda_fail(e, "cudaStreamIsCapturing");
            if (cs != cudaStreamCaptureStatusNone) return ANVIL_ERR_WORKSPACE;
            if (w.ptr) {
                if ((e = cudaFree(w.ptr))) return cuda_fail(e, "cudaFree");
                w.ptr = nullptr;
                w.bytes = 0;
            }
            if ((e = cudaMalloc(&w.ptr, need))) {
                w.ptr = nullptr;
                return cuda_fail(e, "cudaMalloc(workspace)");
            }
            w.bytes = need;
        }
        ws = w.ptr;
    }
    return run_step(&b, 1, nullptr, maps, nmaps, margin, eps, ws, need,
                    static_cast<cudaStream_t>(stream), nullptr);
}

anvil_status anvil_device_error(int clear) {
    DeviceState* dev = nullptr;
    anvil_status st = device_setup(&dev);
    if (st != ANVIL_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned word = 0;
    if ((e = cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost)))
        return cuda_fail(e, "read error word");
    if (clear && (e = cudaMemset(dev->err, 0, sizeof(unsigned))))
        return cuda_fail(e, "clear error word");
    if (clear && (e = cudaDeviceSynchronize())) return cuda_fail(e, "cudaDeviceSynchronize");
    return (word & DEVERR_TIMEOUT) ? ANVIL_ERR_TIMEOUT : ANVIL_OK;
}

anvil_status anvil_last_device_error(void* stream) {
    DeviceState* dev = nullptr;
    anvil_status st = device_setup(&dev);
    if (st != ANVIL_OK) return st;
    unsigned word = 0;
    cudaError_t e = read_error_word_on_stream(dev->err, 1, &word, static_cast<cudaStream_t>(stream));
    if (e) return cuda_fail(e, "read error word");
    return (word & DEVERR_TIMEOUT) ? ANVIL_ERR_TIMEOUT : ANVIL_OK;
}

anvil_status anvil_selftest_wait_timeout(unsigned timeout_us, void* stream) {
    DeviceState* dev = nullptr;
    anvil_status st = device_setup(&dev);
    if (st != ANVIL_OK) return st;
    if (timeout_us == 0 || timeout_us > 10000000u) return ANVIL_ERR_INVALID_ARG;
    cudaError_t e = launch_wait_selftest(timeout_us, dev->err, static_cast<cudaStream_t>(stream));
    return e ? cuda_fail(e, "selftest launch") : ANVIL_OK;
}

anvil_status anvil_profile_begin(int max_records) {
    if (max_records < 1 || max_records > (1 << 20)) return ANVIL_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.active) return ANVIL_ERR_INVALID_ARG;
    g_prof.ev = new cudaEvent_t[2 * static_cast<size_t>(max_records)];
    g_prof.kind = new int[max_records];
    for (int i = 0; i < 2 * max_records; ++i) {
        cudaError_t e = cudaEventCreate(&g_prof.ev[i]);
        if (e) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
            delete[] g_prof.ev;
            delete[] g_prof.kind;
            g_prof.ev = nullptr;
            g_prof.kind = nullptr;
            return cuda_fail(e, "cudaEventCreate");
        }
    }
    g_prof.cap = max_records;
    g_prof.used = 0;
    g_prof.active = true;
    return ANVIL_OK;
}

int anvil_profile_end(anvil_profile_record* records, int cap) {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (!g_prof.active) return 0;
    int n = g_prof.used, rc = n;
    for (int i = 0; i < n; ++i) {
        cudaError_t e = cudaEventSynchronize(g_prof.ev[2 * i + 1]);
        float ms = 0.f;
        if (!e) e = cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]);
        if (e) {
            cuda_fail(e, "profile events");
            rc = -1;
            break;
        }
        if (records && i < cap) {
            records[i].kind = g_prof.kind[i];
            records[i].ms = ms;
        }
    }
    for (int i = 0; i < 2 * g_prof.cap; ++i) cudaEventDestroy(g_prof.ev[i]);
    delete[] g_prof.ev;
    delete[] g_prof.kind;
    g_prof.ev = nullptr;
    g_prof.kind = nullptr;
    g_prof.active = false;
    g_prof.cap = g_prof.used = 0;
    return rc;
}

const char* anvil_status_string(anvil_status s) {
    switch (s) {
        case ANVIL_OK: return "ANVIL_OK";
        case ANVIL_ERR_INVALID_ARG: return "ANVIL_ERR_INVALID_ARG";
        case ANVIL_ERR_UNSUPPORTED_SHAPE: return "ANVIL_ERR_UNSUPPORTED_SHAPE";
        case ANVIL_ERR_ALIGNMENT: return "ANVIL_ERR_ALIGNMENT";
        case ANVIL_ERR_ALIAS: return "ANVIL_ERR_ALIAS";
        case ANVIL_ERR_WORKSPACE: return "ANVIL_ERR_WORKSPACE";
        case ANVIL_ERR_CUDA: return "ANVIL_ERR_CUDA";
        case ANVIL_ERR_TIMEOUT: return "ANVIL_ERR_TIMEOUT";
        case ANVIL_ERR_DEVICE: return "ANVIL_ERR_DEVICE";
        case ANVIL_ERR_UNAVAILABLE: return "ANVIL_ERR_UNAVAILABLE";
    }
    return "ANVIL_ERR_UNKNOWN";
}

const char* anvil_last_cuda_error(void) { return g_last_error; }

anvil_status anvil_timeline_read(void* host, size_t bytes) {
    if (!host || !bytes) return ANVIL_ERR_INVALID_ARG;
    const cudaError_t e = timeline_copy(host, bytes, 0);
    if (e == cudaErrorNotSupported) return ANVIL_ERR_UNAVAILABLE;
    return e ? cuda_fail(e, "timeline read") : ANVIL_OK;
}

anvil_status anvil_timeline_clear(void) {
    const cudaError_t e = timeline_copy(nullptr, 0, 1);
    if (e == cudaErrorNotSupported) return ANVIL_ERR_UNAVAILABLE;
    return e ? cuda_fail(e, "timeline clear") : ANVIL_OK;
}

anvil_status anvil_bank_step_noalloc(const float* grad, float* velocity, int g, int m, int n,
                                     float momentum, float fast_beta, float fast_weight,
                                     float slow_beta, const anvil_map* maps, int nmaps,
                                     float margin, float eps, uint16_t* out, void* stream) {
    anvil_bank_desc b;
    b.grad = grad;
    b.velocity = velocity;
    b.out = out;
    b.g = g;
    b.m = m;
    b.n = n;
    b.scalars.momentum = momentum;
    b.scalars.fast_beta = fast_beta;
    b.scalars.fast_weight = fast_weight;
    b.scalars.slow_beta = slow_beta;
    b.grad_bf16 = 0;
    b.tail_link = nullptr;
    if (!maps) {
        maps = kAnvilMaps;
        nmaps = 6;
    }
    anvil_status st;
    const size_t need = checked_layout_bytes(&b, maps, nmaps, &st);
    if (st != ANVIL_OK) return st;
    if (need > ANVIL_STATIC_SCRATCH_BYTES) {
        snprintf(g_last_error, sizeof(g_last_error),
                 "anvil_bank_step_noalloc: %d x %d x %d needs %zu bytes of scratch; the fixed "
                 "scratch holds %zu",
                 g, m, n, need, static_cast<size_t>(ANVIL_STATIC_SCRATCH_BYTES));
        return ANVIL_ERR_WORKSPACE;
    }
    DeviceState* ds = nullptr;
    if ((st = device_setup(&ds)) != ANVIL_OK) return st;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return ANVIL_ERR_DEVICE;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mutex);
        if (!g_static_addr[dev]) {
            // once per GPU, with that GPU current: the array's device address
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_static_scratch);
            if (e != cudaSuccess || !ptr)
                return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol,
                                 "cudaGetSymbolAddress(fixed scratch)");
            g_static_addr[dev] = ptr;
        }
        scratch = g_static_addr[dev];
    }
    // Every byte of the scratch that the step reads is written earlier in the same step,
    // so what a previous call left there does not matter.
    return run_step(&b, 1, nullptr, maps, nmaps, margin, eps, scratch,
                    static_cast<size_t>(ANVIL_STATIC_SCRATCH_BYTES),
                    static_cast<cudaStream_t>(stream), nullptr);
}

int anvil_schedule_runs(const anvil_bank_desc* banks, int nbanks, int nmaps, anvil_schedule_run* runs,
                        int cap) {
    if (nmaps < 1 || nmaps > ANVIL_MAX_MAPS || cap < 0 || (cap > 0 && !runs)) return -1;
    Layout L;
    if (make_layout(banks, nbanks, &L) != ANVIL_OK) return -1;
    CascadeParams* cp = new (std::nothrow) CascadeParams;
    if (!cp) return -1;
    memset(cp, 0, sizeof(*cp));
    int order[ANVIL_MAX_BANKS];
    cascade_bank_order(L.bank, nbanks, order);
    for (int q = 0; q < nbanks; ++q) {
        const Geom& G = L.bank[order[q]];
        CascadeBank& cb = cp->bank[q];
        cb.g = G.g;
        cb.s_pad = G.s_pad;
        cb.L_pad = G.L_pad;
        cb.m = G.m;
        cb.n = G.n;
        cb.tall = G.tall;
        cb.T = G.s_pad / PAIR;
        cb.ntl = G.L_pad / PAIR;
        cb.mat_begin = G.mat_begin;
    }
    cp->nbanks = nbanks;
    anvil_map maps[ANVIL_MAX_MAPS];
    for (int k = 0; k < nmaps; ++k) maps[k] = anvil_map{1.f, 0.f, 0.f};  // coefficients do not shape the order
    build_phases(cp, maps, nmaps);
    order_phase_major(cp, nullptr);
    const int nruns = cp->nruns;
    for (int r = 0; r < nruns && r < cap; ++r) {
        const CascadeRun& R = cp->run[r];
        const CascadeBank& cb = cp->bank[R.bank];
        runs[r].phase = R.phase;
        runs[r].op = cp->phase[R.phase].op;
        runs[r].bank = order[R.bank];
        runs[r].mat0 = R.mat0;
        runs[r].nmat = static_cast<int>(R.nmat);
        runs[r].begin = R.begin;
        runs[r].tiles = phase_tiles(cb, cp->phase[R.phase].op);
    }
    delete cp;
    return nruns;
}

}  // extern "C"
