// anvil_device.cuh -- sm_103a device helpers: bf16 rounding, mbarriers with bounded
// waits, TMA tensor loads, and the tcgen05 (5th-generation tensor core) MMA / TMEM
// instructions, all as inline PTX.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "anvil_internal.h"

namespace anvil {

// A bounded wait gives up after this long (a healthy wait here lasts microseconds).
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- bf16 (round to nearest even, CUDA's conversion) --------------------------------
__device__ __forceinline__ uint16_t f2bf(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf2f(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ float round_bf(float x) { return bf2f(f2bf(x)); }

// ---- packed pairs: two fp32 in one 64-bit register (element 0 in the low half), and two
// bf16 in one 32-bit word (element 0 in the low half).  The f32x2 operations are two
// independent IEEE round-to-nearest operations.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    return (static_cast<uint64_t>(__float_as_uint(hi)) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Negation of both halves (exact).  A difference a - b is taken as f2_add(a, f2_neg(b)):
// a packed subtract whose operand is a packed product was measured to come out as one
// fused rounding (1 ulp off in about 2.4% of elements), the addition of the negated product
// as two roundings, like the scalar operations.
__device__ __forceinline__ uint64_t f2_neg(uint64_t a) { return a ^ 0x8000000080000000ull; }
// two bf16 (round to nearest even) of a packed fp32 pair
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(d)
        : "f"(__uint_as_float(static_cast<uint32_t>(v >> 32))),
          "f"(__uint_as_float(static_cast<uint32_t>(v))));
    return d;
}
// packed fp32 pair of two bf16 (exact)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
    return (static_cast<uint64_t>(w & 0xffff0000u) << 32) | (w << 16);
}

// bf16(RN(x / dd)) for four pairs of fp32 x, given rcp2 = (RN(1/dd), RN(1/dd)).  The
// product q = RN(x * RN(1/dd)) is within 2.5 ulp of RN(x / dd), so both round to the same
// bf16 unless a bf16 rounding boundary (low 16 bits 0x8000) lies within 8 ulps of q, or q
// is tiny (exponent < 8), huge or not finite; a chunk with such an element (about one in
// 1000) takes the correctly rounded division, out of line.
__device__ __forceinline__ bool near_bf16_boundary(uint32_t b) {
    return (((b + 8u) & 0xfff0u) == 0x8000u) | ((((b >> 23) + 1u) & 0xffu) < 9u);
}
static __device__ __noinline__ uint4 div4_exact(uint64_t x0, uint64_t x1, uint64_t x2, uint64_t x3, float dd) {
    const uint64_t x[4] = {x0, x1, x2, x3};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = f2_to_bf2(f2_pack(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(x[e])), dd),
                                 __fdiv_rn(__uint_as_float(static_cast<uint32_t>(x[e] >> 32)), dd)));
    return make_uint4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ uint4 div4_to_bf2(uint64_t x0, uint64_t x1, uint64_t x2, uint64_t x3, uint64_t rcp2,
                                             float dd) {
    const uint64_t q0 = f2_mul(x0, rcp2), q1 = f2_mul(x1, rcp2), q2 = f2_mul(x2, rcp2), q3 = f2_mul(x3, rcp2);
    const bool near = near_bf16_boundary(static_cast<uint32_t>(q0)) | near_bf16_boundary(static_cast<uint32_t>(q0 >> 32)) |
                      near_bf16_boundary(static_cast<uint32_t>(q1)) | near_bf16_boundary(static_cast<uint32_t>(q1 >> 32)) |
                      near_bf16_boundary(static_cast<uint32_t>(q2)) | near_bf16_boundary(static_cast<uint32_t>(q2 >> 32)) |
                      near_bf16_boundary(static_cast<uint32_t>(q3)) | near_bf16_boundary(static_cast<uint32_t>(q3 >> 32));
    if (__builtin_expect(near, 0)) return div4_exact(x0, x1, x2, x3, dd);
    return make_uint4(f2_to_bf2(q0), f2_to_bf2(q1), f2_to_bf2(q2), f2_to_bf2(q3));
}

// ---- programmatic dependent launch ---------------------------------------------------
// A kernel launched with programmatic stream serialisation may start while the previous
// kernel of the stream finishes; it must wait here before touching anything that kernel
// writes or reads.  Without that launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait_previous() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel of the stream be scheduled (it still waits for this one to finish
// before it touches memory).
__device__ __forceinline__ void pdl_allow_next() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- mbarrier -----------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
// Makes the barrier initialisation visible to the async proxy (TMA, tcgen05.commit).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrival that orders nothing before it (a pure progress signal).
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// 16-byte shared-memory load / store at a shared-window address.
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Non-blocking test of the phase with this parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits until the phase with this parity completes, or gives up after `limit_ns`,
// recording DEVERR_TIMEOUT.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, DEVERR_TIMEOUT);
            return false;
        }
    }
}

// ---- TMA ------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}
// 3-D tiled load of one box into shared memory; completion is signalled on `bar`
// as transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 3-D tiled store of one box from shared memory (bulk async-group completion).
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            tmap),
        "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// tma_store_3d with an L2 evict-last policy on the stored lines (data that the next
// phases read again).
__device__ __forceinline__ void tma_store_3d_keep(const void* tmap, const void* smem_src, int c0, int c1, int c2) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], pol;\n\t}"
        ::"l"(tmap), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk store has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until all but the most recent committed bulk store have finished reading their
// shared-memory sources.
__device__ __forceinline__ void bulk_wait_read_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Waits until every committed bulk store but the two most recent has completed.
__device__ __forceinline__ void bulk_wait_all_but_two() {
    asm volatile("cp.async.bulk.wait_group 2;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Barrier over a subset of the CTA's warps (id 1..15; `count` threads, a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier over `count` threads that also ORs a flag across them: every thread gets
// the same answer, so a group can leave a loop together.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.cta.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(flag ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---- clusters (2-CTA pairs) -------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// Arrive on an mbarrier given by its cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// All threads of both CTAs of the cluster.
// Bounded wait with cluster-scope acquire, for a barrier that a peer CTA's thread arrives
// on (after writing the data it guards into this CTA's shared memory).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, unsigned* err,
                                                  unsigned long long limit_ns = WAIT_LIMIT_NS) {
    const uint32_t a = smem_u32(bar);
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
        if (i == 0) t0 = globaltimer_ns();
        else if ((i & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            atomicOr(err, DEVERR_TIMEOUT);
            return false;
        }
    }
}
// 32-bit store into a CTA of the cluster (address from map_to_rank).
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// 16-byte store into a CTA of the cluster (address from map_to_rank).
__device__ __forceinline__ void st_cluster_v4(uint32_t cluster_addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// TMA load into this CTA's shared memory whose completion is counted on an mbarrier of
// the CTA pair (here: the leader CTA's), given by its cluster address.
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const void* tmap, uint32_t bar_cluster,
                                                 int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ---- tcgen05 for CTA pairs (.cta_group::2): one warp of EACH CTA of the pair allocates
// and frees (the columns are the same in both); only the leader CTA issues MMAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (M = 256 across the pair: 128 rows in each CTA's TMEM) (+)= A * B^T, with A split
// by rows and B split by columns between the two CTAs' shared memory (same offsets).
__device__ __forceinline__ void umma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on the barrier at this address in every CTA of `cta_mask` when all
// previously issued MMAs of this thread complete.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---- tcgen05: TMEM allocation ----------------------------------------------------------
// Executed by one full warp.  The allocated column base is written to *slot (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- tcgen05: shared-memory matrix descriptors ------------------------------------------
// The 64-bit descriptor: start address >> 4 in bits 0-13, leading-dimension byte
// offset >> 4 in bits 16-29, stride-dimension byte offset >> 4 in bits 32-45, the
// fixed value 1 in bits 46-47, base offset 0 (every swizzle atom here starts on a
// 1024-byte boundary), swizzle mode in bits 61-63 (2 = 128-byte swizzle).
//   K-major, 128-byte swizzle: rows of 64 bf16 (128 B), 8-row groups SBO apart;
//     LBO unused.  A k-step of 16 elements inside the row advances the start by 32 B.
//   MN-major, 128-byte swizzle: 64 contiguous MN elements per 128-byte row, one row
//     per k; 8-row k groups SBO apart, 64-element MN chunks LBO apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// The same descriptor in two halves, for the MMA issuer's inner loop: the high word (stride
// offset 1024 bytes, the fixed 1, 128-byte swizzle) is common to every operand here, and
// the low word (start address >> 4, leading offset >> 4) advances by a k-step's bytes >> 4.
constexpr uint32_t SW128_DESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t sw128_desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
    return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t lo) {
    return (static_cast<uint64_t>(SW128_DESC_HI) << 32) | lo;
}

// Instruction descriptor of tcgen05.mma .kind::f16 with bf16 A and B, fp32 accumulate:
// D format (bits 4-5) = 1 (f32), A format (7-9) = 1 (bf16), B format (10-12) = 1 (bf16),
// A major (15) and B major (16): 0 = K-major, 1 = MN-major, N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by a single thread.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every tcgen05.mma this thread issued before it completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp gets lane (base + t).
// The wait is in the same asm statement, so no register is read before it lands.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace anvil
