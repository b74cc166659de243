// anvil_gemm.cu -- the ANVIL cascade (page "modded-nanogpt track_1_short/optim/anvil.py",
// anvil_cascade: the XTX / XXT, ba_plus_cAA and baddbmm steps of every spectral map) as ONE
// persistent tcgen05 kernel for sm_103a that walks every phase of a step:
//
//   OP_GRAM_NORM : A  = bf16(bf16(Y Y^T) / d^2)     (the first Gram, on X_raw)
//   OP_GRAM      : A  = bf16(Y Y^T)
//   OP_SQPOLY    : B  = bf16(b A + c A A)
//   OP_XUPDATE   : Y' = bf16(a Y + B Y)             (OP_XUPDATE_OUT: the last, into out)
//
// in the small-side-major layout of anvil_internal.h.  A and B are symmetric: the Gram
// and A A compute and store only the diagonal and upper 256x256 blocks, and a product
// operand's k-block left of its diagonal block is read, MN-major, from the transposed
// upper block.  A A contracts A's rows with A's rows (A A = A A^T), so every operand is
// K-major except those mirrored k-blocks and Y in the X-update.
//
// Work items.  An item is one 256x256 output tile of one matrix in one phase.  The host
// numbers the items by a list of runs (each: one phase of a range of matrices of one
// bank) and the persistent grid of CTA pairs takes them in list order: a pair's scheduler
// warp takes the next item from a global counter, so each pair's items increase.  Every
// finished tile adds to a per-matrix completion counter in global memory (a release add,
// once the tile's stores have landed, from a publisher warp, so that no epilogue thread
// waits for its own stores to drain).  The scheduler hands an item to the pair's other
// roles only once its matrix's counters reach the totals its phase needs (acquire), as a
// resolved entry (phase, matrix, block, k-blocks, operand maps) in shared memory: the
// producer and the MMA issuer, whose work is the critical path, read nothing else at an
// item boundary.  A pair therefore moves on to the next phase of one matrix while other
// matrices are still in the previous one, with no kernel boundary between the phases.
// Each phase of a matrix reads only what the phases before it wrote and waits for all of
// them, which also orders every reuse of the A, B and Y buffers.  Every entry in a ring
// can complete without another pair, an epilogue publishes its last tile before it waits
// for an entry, and the lowest-numbered unfinished item never waits, so the walk always
// progresses (every pair of the grid is co-resident: one CTA per SM).
//
// CTA pairs.  Clusters of two CTAs on two SMs compute a tile with tcgen05.mma.cta_group::2
// (M = 256, N = 256, K = 16): CTA rank r loads rows 128r.. of the tile's A operand and
// columns 128r.. of its B operand (TMA, completions counted on the leader's barrier) and
// holds output rows 128r.. in its TMEM.  Warp 0 (one lane) issues the TMA loads into a
// 5-stage ring; warp 1 allocates 512 TMEM columns in both CTAs and, in the leader only,
// issues the MMAs into one of two 256-column accumulators, committing to both CTAs'
// barriers; warps 2-9 (two groups of four, one per column half) run the fused epilogue on
// the other accumulator; warp 10 publishes finished tiles; warp 11 (leader CTA) is the
// pair's scheduler.  The epilogue input tile (A for B = bA + cAA, Y for the X-update)
// arrives by TMA into 128x64 boxes (128-byte swizzle), is updated
// in place with packed f32x2 arithmetic and leaves by TMA store; the X^T output of tall
// banks leaves as plain stores, 64 contiguous bytes per warp.
//
// Every wait is bounded (anvil_device.cuh): a wait that gives up sets the device error
// word and an abort flag; all roles stop, in-flight copies and MMAs are waited for
// (bounded), the TMEM is freed and the CTA exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include "anvil_device.cuh"
#include "anvil_internal.h"

namespace anvil {

constexpr int SMEM_MAX = 227 * 1024;    // opt-in dynamic shared memory per block
constexpr int QBOX = TILE * 64 * 2;     // one 128 x 64 bf16 staging box (16 KB)
constexpr int NBOX = 4;                 // staging boxes: one per quarter of a CTA's tile
constexpr int A_STAGE = TILE * BK * 2;  // 16 KB: this CTA's A rows of a k-block
constexpr int B_STAGE = TILE * BK * 2;  // 16 KB: this CTA's B half of a k-block
constexpr int STAGE = A_STAGE + B_STAGE;
constexpr int STAGES = (SMEM_MAX - 2048 - NBOX * QBOX) / STAGE;  // 5
constexpr int GEMM_SMEM = STAGES * STAGE + NBOX * QBOX + 1024;   // + alignment slack
constexpr int BN = PAIR;     // output columns per CTA
constexpr int NQ = BN / 64;  // quarters (64 columns) per tile
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int EPI_GROUPS = 2;
constexpr int PUB_DEPTH = 4;  // completion messages in flight per epilogue group
// warp 0: TMA producer; warp 1: TMEM owner and MMA issuer; warps 2-9: epilogue, in two
// groups of four (one warp per TMEM lane quadrant), group h owning quarters 2h, 2h+1;
// warp 10: publisher of finished tiles; warp 11: the pair's item scheduler (leader CTA).
constexpr int PUB_WARP = 2 + EPI_GROUPS * 4;
constexpr int SCHED_WARP = PUB_WARP + 1;
constexpr int GEMM_THREADS = 32 * (SCHED_WARP + 1);

// Per-item timeline (only in a library built with -DANVIL_TIMELINE; the macro is empty
// otherwise and its arguments are not evaluated).  Item t of a launch owns TL_FIELDS
// 64-bit words, written by the leader CTA of the pair that ran it (TL_* field names in
// anvil_internal.h): %globaltimer nanoseconds at each hand-off, SM cycles around the
// k-loop.
#ifdef ANVIL_TIMELINE
__device__ unsigned long long g_timeline[TL_ITEMS * TL_FIELDS];
#define TL_PUT(t, k, v)                                                              \
    do {                                                                             \
        const int tl_t_ = (t);                                                       \
        if (tl_t_ >= 0 && tl_t_ < TL_ITEMS) g_timeline[tl_t_ * TL_FIELDS + (k)] = (v); \
    } while (0)
#else
#define TL_PUT(t, k, v) \
    do {                \
    } while (0)
#endif

__host__ __device__ constexpr bool op_sym(int op) {
    return op == OP_GRAM || op == OP_GRAM_NORM || op == OP_SQPOLY;
}
__host__ __device__ constexpr bool op_xupdate(int op) {
    return op == OP_XUPDATE || op == OP_XUPDATE_OUT;
}
__host__ __device__ constexpr bool op_gram(int op) { return op == OP_GRAM || op == OP_GRAM_NORM; }

struct Item {
    int ph, bank, mat, bi, bj;
};

// Item schedule of a CTA pair: the leader's scheduler warp takes the pair's next item
// from the launch's global counter (an atomic add), decodes it, waits until the phases
// it reads are complete for its matrix, and writes the resolved entry (a Work) into a
// ring in both CTAs' shared memory; every role of both CTAs reads the ring in order and
// frees each slot on the leader's barrier.  Items thus go to whichever pair is ready for
// work, in list order, and each pair's items increase; no role but the scheduler reads
// the kernel parameters or the completion counters at an item boundary.  The writes need
// release semantics, which make a thread wait for its own asynchronous copies; the
// scheduler has none, and the readers free slots with relaxed arrivals (ordered after
// their reads of the slot by a data dependency).
constexpr int SDEPTH = 6;                         // ring slots
constexpr int SAHEAD = 3;                         // entries the scheduler may run ahead of the producer
constexpr int SCONSUMERS = 3 + 2 * EPI_GROUPS;    // both producers, the MMA, every epilogue group

// A resolved item: two 16-byte words.
//   w0 = {t, op | bank << 8 | ph << 16, mat, nkb}    (t >= the item count: no more work)
//   w1 = {bi, bj, the operand map slots (map_a, map_a_t, map_b, map_b_t: one byte each), check}
// where check = ~(the XOR of the other seven words), so that the XOR of all eight is
// 0xffffffff: a reader derives its arrival count from it, which makes the arrival depend
// on every word it read (see sched_take).
struct Work {
    uint4 w0, w1;
    __device__ int t() const { return static_cast<int>(w0.x); }
    __device__ int op() const { return static_cast<int>(w0.y & 0xffu); }
    __device__ int bank() const { return static_cast<int>((w0.y >> 8) & 0xffu); }
    __device__ int ph() const { return static_cast<int>(w0.y >> 16); }
    __device__ int mat() const { return static_cast<int>(w0.z); }
    __device__ int nkb() const { return static_cast<int>(w0.w); }
    __device__ int bi() const { return static_cast<int>(w1.x); }
    __device__ int bj() const { return static_cast<int>(w1.y); }
    __device__ int map(int k) const { return static_cast<int>(static_cast<int8_t>((w1.z >> (8 * k)) & 0xffu)); }
    // A diagonal block of a symmetric product (a Gram or A*A block with bi == bj): in each
    // CTA the A rows and the B columns are the same operand rows, read through the same
    // maps, so one load serves both descriptors.
    __device__ bool shared_ab() const {
        return !op_xupdate(op()) && w1.x == w1.y && ((w1.z ^ (w1.z >> 16)) & 0xffffu) == 0u;
    }
};

struct alignas(16) SchedRing {
    uint4 work[SDEPTH][2];   // read and written as 16-byte words: 16-byte aligned
    uint64_t full[SDEPTH];   // slot written (this CTA)
    uint64_t empty[SDEPTH];  // slot read by every consumer (leader CTA)
    uint64_t taken[SDEPTH];  // slot read by the leader's producer (leader CTA)
};

static_assert(offsetof(SchedRing, work) == 0 && alignof(SchedRing) == 16, "ring words need 16-byte alignment");

// Scheduler: publishes w as the k-th entry.
__device__ __forceinline__ bool sched_push(SchedRing& q, int k, const Work& w, unsigned* err) {
    const int s = k % SDEPTH;
    if (!mbar_wait_cluster(&q.empty[s], ((k / SDEPTH) & 1) ^ 1, err)) return false;
    sts128(smem_u32(&q.work[s][0]), w.w0);
    sts128(smem_u32(&q.work[s][1]), w.w1);
    st_cluster_v4(map_to_rank(&q.work[s][0], 1), w.w0);
    st_cluster_v4(map_to_rank(&q.work[s][1], 1), w.w1);
    mbar_arrive_cta(&q.full[s]);
    mbar_arrive_cluster(map_to_rank(&q.full[s], 1));
    return true;
}

// Any other role: the k-th entry (t = INT_MAX if the wait gave up).
__device__ __forceinline__ Work sched_take(SchedRing& q, int k, unsigned* err) {
    const int s = k % SDEPTH;
    Work w;
    if (!mbar_wait_cluster(&q.full[s], (k / SDEPTH) & 1, err)) {
        w.w0 = make_uint4(0x7fffffffu, 0u, 0u, 0u);
        w.w1 = make_uint4(0u, 0u, 0u, 0u);
        return w;
    }
    w.w0 = lds128(smem_u32(&q.work[s][0]));
    w.w1 = lds128(smem_u32(&q.work[s][1]));
    // the arrival count, 1, is computed from every word read (their XOR is 0xffffffff), so
    // the relaxed arrival cannot overtake the reads of the slot it frees
    const uint32_t all = w.w0.x ^ w.w0.y ^ w.w0.z ^ w.w0.w ^ w.w1.x ^ w.w1.y ^ w.w1.z ^ w.w1.w;
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                     map_to_rank(&q.empty[s], 0)),
                 "r"(all >> 31)
                 : "memory");
    return w;
}

// Item t (an index into the call's item list) -> phase, bank, matrix, block row and
// column: the run holding t (binary search over this launch's runs), then the tile.
__device__ __forceinline__ Item decode_item(const CascadeParams& p, int t) {
    int lo = p.first_run, hi = p.end_run - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.run[mid].begin <= t) lo = mid;
        else hi = mid - 1;
    }
    const CascadeRun& R = p.run[lo];
    const CascadePhase& P = p.phase[R.phase];
    const CascadeBank& B = p.bank[R.bank];
    Item it;
    it.ph = R.phase;
    it.bank = R.bank;
    const int T = B.T;
    const bool sym = op_sym(P.op);
    const int tpm = sym ? T * (T + 1) / 2 : T * B.ntl;
    const int local = t - R.begin;
    const int lm = local / tpm;
    it.mat = R.mat0 + lm;
    int r = local - lm * tpm;
    if (sym) {
        int ti = 0;
        while (r >= T - ti) {
            r -= T - ti;
            ++ti;
        }
        it.bi = ti;
        it.bj = ti + r;
    } else {
        it.bi = r / B.ntl;
        it.bj = r - it.bi * B.ntl;
    }
    return it;
}

__device__ __forceinline__ void work_seal(Work& w) {
    w.w1.w = ~(w.w0.x ^ w.w0.y ^ w.w0.z ^ w.w0.w ^ w.w1.x ^ w.w1.y ^ w.w1.z);
}

// The resolved entry of item t of this launch (t >= nitems: the end marker).
__device__ __forceinline__ Work make_work(const CascadeParams& p, int item0, int nitems, int t) {
    Work w;
    w.w0 = make_uint4(static_cast<uint32_t>(t), 0u, 0u, 0u);
    w.w1 = make_uint4(0u, 0u, 0u, 0u);
    if (t >= nitems) {
        work_seal(w);
        return w;
    }
    const Item c = decode_item(p, item0 + t);
    const CascadePhase& P = p.phase[c.ph];
    const CascadeBank& bk = p.bank[c.bank];
    const int nkb = (op_gram(P.op) ? bk.L_pad : bk.s_pad) / BK;
    w.w0 = make_uint4(static_cast<uint32_t>(t), static_cast<uint32_t>(P.op | (c.bank << 8) | (c.ph << 16)),
                      static_cast<uint32_t>(c.mat), static_cast<uint32_t>(nkb));
    const uint32_t maps = (static_cast<uint32_t>(P.map_a) & 0xffu) | ((static_cast<uint32_t>(P.map_a_t) & 0xffu) << 8) |
                          ((static_cast<uint32_t>(P.map_b) & 0xffu) << 16) |
                          ((static_cast<uint32_t>(P.map_b_t) & 0xffu) << 24);
    w.w1 = make_uint4(static_cast<uint32_t>(c.bi), static_cast<uint32_t>(c.bj), maps, 0u);
    work_seal(w);
    return w;
}

__device__ __forceinline__ Item work_item(const Work& w) {
    Item c;
    c.ph = w.ph();
    c.bank = w.bank();
    c.mat = w.mat();
    c.bi = w.bi();
    c.bj = w.bj();
    return c;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Whether the phases item `it` reads are complete for its matrix (no wait).
__device__ __forceinline__ bool deps_ready(const CascadeParams& p, const Item& it) {
    const CascadePhase& P = p.phase[it.ph];
    const unsigned nc = P.need_chain[it.bank];
    return !nc || ld_acquire(p.chain + p.bank[it.bank].mat_begin + it.mat) >= nc;
}

// Waits (bounded) for the same; then orders this thread's later TMA loads after it.
__device__ __forceinline__ bool deps_wait(const CascadeParams& p, const Item& it) {
    if (!deps_ready(p, it)) {
        const unsigned long long t0 = globaltimer_ns();
        for (uint32_t i = 1;; ++i) {
            __nanosleep(100);
            if (deps_ready(p, it)) break;
            if ((i & 15u) == 0 && globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                atomicOr(p.err, DEVERR_TIMEOUT);
                return false;
            }
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// This CTA's operand boxes of k-block kb of entry w, loaded by TMA into the stage at `sa`
// (both CTAs' bytes complete on the leader's barrier `fb`).  CTA rank r holds rows 128r..
// of the tile's A operand and columns 128r.. of its B operand.  A k-block left of a
// symmetric operand's diagonal block comes from the upper block it mirrors, read MN-major
// as two 64 x 64 boxes (k rows, operand rows); the X-update's Y is MN-major too: Y rows
// kb*64 .. +63, this CTA's 128 columns in two 64-column boxes, 8 KB apart.
__device__ __forceinline__ void load_kblock(const CascadeParams& p, const Work& w, int kb, uint32_t rank,
                                            uint8_t* sa, uint32_t fb) {
    const CUtensorMap* tm = p.bank[w.bank()].tm;
    const int bi = w.bi(), bj = w.bj(), mat = w.mat();
    const int arow = bi * PAIR + TILE * static_cast<int>(rank);
    const int bofs = bj * PAIR + TILE * static_cast<int>(rank);
    const int map_a = w.map(0), map_a_t = w.map(1), map_b = w.map(2), map_b_t = w.map(3);
    uint8_t* sb = sa + A_STAGE;
    const bool shared = w.shared_ab();
    if (map_a_t >= 0 && kb * BK < bi * PAIR) {
        tma_load_3d_pair(sa, &tm[map_a_t], fb, arow, kb * BK, mat);
        tma_load_3d_pair(sa + 8192, &tm[map_a_t], fb, arow + 64, kb * BK, mat);
    } else {
        tma_load_3d_pair(sa, &tm[map_a], fb, kb * BK, arow, mat);
    }
    const bool xu = op_xupdate(w.op());
    if (shared) return;
    if (xu || (map_b_t >= 0 && kb * BK < bj * PAIR)) {
        const CUtensorMap* tb = &tm[xu ? map_b : map_b_t];
        tma_load_3d_pair(sb, tb, fb, bofs, kb * BK, mat);
        tma_load_3d_pair(sb + 8192, tb, fb, bofs + 64, kb * BK, mat);
    } else {
        tma_load_3d_pair(sb, &tm[map_b], fb, kb * BK, bofs, mat);
    }
}

// The completion counter a finished tile adds to.
__device__ __forceinline__ unsigned* tile_counter(const CascadeParams& p, const Item& it) {
    return p.chain + p.bank[it.bank].mat_begin + it.mat;
}

// The elementwise part of each op's epilogue on a pair: accumulator values v (packed fp32
// pair) and input word xw (two bf16); returns two bf16.  Each product and sum is rounded
// on its own (the page's fp32 tensor operations one at a time).  (The first Gram's
// quotient is taken four pairs at a time, div4_to_bf2.)
template <int OP>
__device__ __forceinline__ uint32_t epi_pair(uint64_t v, uint32_t xw, uint64_t coef_x, uint64_t coef_v) {
    if (OP == OP_GRAM) return f2_to_bf2(v);
    const uint64_t t = f2_mul(coef_x, bf2_to_f2(xw));                     // b A  or  a Y
    if (OP == OP_SQPOLY) return f2_to_bf2(f2_add(t, f2_mul(coef_v, v)));  // + c acc
    return f2_to_bf2(f2_add(t, v));                                       // + acc
}

__device__ __forceinline__ uint16_t half_of(const uint32_t (&o)[4], int e) {
    return static_cast<uint16_t>((e & 1) ? (o[e >> 1] >> 16) : (o[e >> 1] & 0xffffu));
}

// Per-thread epilogue state of one group.
struct EpiCtx {
    uint8_t* stg;        // staging boxes
    uint64_t* epi_bar;   // input-load barriers, one per quarter
    int r;               // row of the CTA's tile this thread owns
    int grp, lane;
    bool leader;         // lane 0 of the group's first warp
    int last_box;        // staging box of the group's latest TMA store (-1: none)
    bool fail;           // one of this thread's waits gave up
    int npub;            // completion messages sent to the publisher
};

// A release add makes this thread wait for its own stores in flight, so the epilogue
// hands each finished tile to the publisher warp instead: the group leader, once the
// tile's TMA stores have completed (and after the group barrier that follows its plain
// stores), writes the counter's address into a mailbox slot and arrives on the slot's
// barrier (release, CTA scope); the publisher acquires it and performs the release add
// at GPU scope.  A null address ends the group's messages.
struct Mailbox {
    uint64_t full[EPI_GROUPS][PUB_DEPTH];
    uint64_t empty[EPI_GROUPS][PUB_DEPTH];
    unsigned* slot[EPI_GROUPS][PUB_DEPTH];
};

__device__ __forceinline__ void send_done(Mailbox& mb, EpiCtx& x, unsigned* cnt, unsigned* err) {
    asm volatile("fence.proxy.async.global;" ::: "memory");  // the tile's TMA stores, then the message
    const int k = x.npub++;
    const int s = k % PUB_DEPTH;
    if (!mbar_wait(&mb.empty[x.grp][s], ((k / PUB_DEPTH) & 1) ^ 1, err)) x.fail = true;
    mb.slot[x.grp][s] = cnt;
    mbar_arrive_cta(&mb.full[x.grp][s]);
}

// The quarters of one product tile that this thread's group owns: read the accumulator
// (tbase: TMEM address of the thread's lane quadrant in the accumulator), combine with
// the input box, store.  tempty: the leader CTA's barrier for this
// accumulator.  A wait that gives up sets x.fail and the tile runs to its end all the
// same (its values are then meaningless), so every thread of the group reaches every
// group barrier.
template <int OP>
__device__ __forceinline__ void epi_tile(const CascadeParams& p, const CascadeBank& bk,
                                         const CascadePhase& P, const Item& c, uint32_t rank,
                                         EpiCtx& x, uint32_t tbase, uint32_t tempty, uint32_t in_phase) {
    constexpr bool has_in = !op_gram(OP);
    const int row0 = c.bi * PAIR + TILE * static_cast<int>(rank);  // this CTA's first row
    const int col0 = c.bj * PAIR;
    const int r = x.r;
    // the direct tile leaves by TMA except the last X-update into an `out` that cannot
    // take it (rows not 16-byte aligned: plain stores); a tall bank's X = Y^T leaves by TMA
    // too, written transposed into the staging box: quarter q of this CTA's 128 rows is
    // out rows col0 + 64q .. +63 by out columns row0 .. row0 + 127, two 64 x 64 boxes of out
    const bool tma_trans = OP == OP_XUPDATE_OUT && bk.tall && bk.out_tma;
    const bool tma_direct = OP != OP_XUPDATE_OUT || (bk.out_tma && !bk.tall);
    uint64_t coef_x = f2_pack(OP == OP_SQPOLY ? P.b : P.a, OP == OP_SQPOLY ? P.b : P.a);
    const uint64_t coef_v = f2_pack(P.c, P.c);
    float dd = 0.f;
    if (OP == OP_GRAM_NORM) {  // coef_x: the reciprocal of d^2 for div4_to_bf2
        const float d = bk.d[c.mat];
        dd = __fmul_rn(d, d);
        const float rcp = __frcp_rn(dd);
        coef_x = f2_pack(rcp, rcp);
    }
    for (int q = 2 * x.grp; q < 2 * x.grp + 2; ++q) {
        int box = q;
        if (!has_in) {
            // a free Gram output box: not the one of the latest store, and every older
            // store has finished reading its box
            box = x.last_box == 2 * x.grp ? 2 * x.grp + 1 : 2 * x.grp;
            if (x.leader) bulk_wait_read_but_one();
            named_barrier_sync(1 + x.grp, 128);
        } else if (!mbar_wait(&x.epi_bar[q], in_phase, p.err)) {
            x.fail = true;
        }
        const uint32_t dbox = smem_u32(x.stg) + static_cast<uint32_t>(box * QBOX);
        const uint32_t drow = dbox + static_cast<uint32_t>(r * 128);
        // transposed output overwrites other threads' input rows: the group reads all of
        // the quarter's input first
        uint4 xall[8];
        if (tma_trans) {
#pragma unroll
            for (int j = 0; j < 8; ++j) xall[j] = lds128(drow + static_cast<uint32_t>((j ^ (r & 7)) << 4));
            named_barrier_sync(1 + x.grp, 128);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            // 16-byte chunk j of this 128-byte row sits at chunk j ^ (r % 8); the chunk's
            // four input loads go out together, ahead of the accumulator read
            uint4 xin[4];
            if (has_in) {
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    xin[w] = tma_trans ? xall[cc * 4 + w]
                                       : lds128(drow + static_cast<uint32_t>(((cc * 4 + w) ^ (r & 7)) << 4));
            }
            float v[32];
            tmem_ld_32x32b_x32(tbase + q * 64 + cc * 32, v);
            const int cb = col0 + q * 64 + cc * 32;  // first column of this chunk
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t xw[4] = {has_in ? xin[w].x : 0u, has_in ? xin[w].y : 0u, has_in ? xin[w].z : 0u,
                                        has_in ? xin[w].w : 0u};
                uint32_t o[4];
                if (OP == OP_GRAM_NORM) {  // bf16(bf16(acc) / d^2)
                    const uint4 r4 = div4_to_bf2(bf2_to_f2(f2_to_bf2(f2_pack(v[8 * w + 0], v[8 * w + 1]))),
                                                 bf2_to_f2(f2_to_bf2(f2_pack(v[8 * w + 2], v[8 * w + 3]))),
                                                 bf2_to_f2(f2_to_bf2(f2_pack(v[8 * w + 4], v[8 * w + 5]))),
                                                 bf2_to_f2(f2_to_bf2(f2_pack(v[8 * w + 6], v[8 * w + 7]))), coef_x, dd);
                    o[0] = r4.x; o[1] = r4.y; o[2] = r4.z; o[3] = r4.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[e] = epi_pair<OP>(f2_pack(v[8 * w + 2 * e], v[8 * w + 2 * e + 1]), xw[e], coef_x, coef_v);
                }
                if (tma_direct)
                    sts128(drow + static_cast<uint32_t>(((cc * 4 + w) ^ (r & 7)) << 4), make_uint4(o[0], o[1], o[2], o[3]));
                if (tma_trans) {
                    // element (r, y) of the quarter: out row y is line y of box r / 64 (128-byte
                    // lines, 16-byte chunk k of line y at k ^ (y % 8)), out column r % 64
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int y = cc * 32 + 8 * w + e;
                        sts16(dbox + static_cast<uint32_t>((r >> 6) * 8192 + y * 128 +
                                                           ((((r & 63) >> 3) ^ (y & 7)) << 4) + (r & 7) * 2),
                              half_of(o, e));
                    }
                }
                const int c8 = cb + 8 * w;  // column of o[0]'s low half
                if (OP == OP_XUPDATE_OUT && !tma_direct && !tma_trans) {
                    uint16_t* out = bk.out + static_cast<size_t>(c.mat) * bk.m * bk.n;
                    if (bk.tall) {
                        // X = Y^T: element (row0 + r, c8 + e) -> out row c8 + e, column row0 + r
                        if (row0 + r < bk.n) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (c8 + e < bk.m)
                                    out[static_cast<size_t>(c8 + e) * bk.n + row0 + r] = half_of(o, e);
                        }
                    } else if (row0 + r < bk.m) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (c8 + e < bk.n)
                                out[static_cast<size_t>(row0 + r) * bk.n + c8 + e] = half_of(o, e);
                    }
                }
            }
        }
        if (q == 2 * x.grp + 1) {
            // the accumulator is free once every epilogue warp of both CTAs has read it
            tc_fence_before();
            __syncwarp();
            if (x.lane == 0) mbar_arrive_cluster(tempty);
        }
        fence_proxy_async_smem();
        named_barrier_sync(1 + x.grp, 128);
        if (tma_direct) {
            if (x.leader) {
                // the next Y stays in L2 ahead of the old one: the next map's Gram, B and
                // X-update read it (an evict-last hint; measured 0.8% off the launch)
                if (OP == OP_XUPDATE)
                    tma_store_3d_keep(&bk.tm[P.map_out], x.stg + box * QBOX, col0 + 64 * q, row0, c.mat);
                else
                    tma_store_3d(&bk.tm[P.map_out], x.stg + box * QBOX, col0 + 64 * q, row0, c.mat);
                bulk_commit_group();
            }
            x.last_box = box;
        } else if (tma_trans) {
            if (x.leader) {
                // out [g, m, n]: column coordinate (innermost) = Y row, row coordinate = Y
                // column; boxes wholly in the padding are skipped, the rest clip at m and n
                for (int h = 0; h < 2; ++h)
                    if (row0 + 64 * h < bk.n && col0 + 64 * q < bk.m)
                        tma_store_3d(&bk.tm[P.map_out], x.stg + box * QBOX + h * 8192, row0 + 64 * h, col0 + 64 * q,
                                     c.mat);
                bulk_commit_group();  // one group per quarter, as on the other paths
            }
            x.last_box = box;
        }
    }
}

__global__ void __launch_bounds__(GEMM_THREADS, 1) cascade_kernel(const __grid_constant__ CascadeParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t mma_done_bar;
    __shared__ __align__(8) uint64_t epi_bar[NQ];  // epilogue input loads, one per quarter
    __shared__ __align__(8) Mailbox mbox;
    __shared__ __align__(16) SchedRing sring;
    // each group's current entry, by iteration parity: the leader writes the next one
    // while the group may still read this one
    __shared__ uint4 grp_work[EPI_GROUPS][2][2];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int aborted;

    pdl_allow_next();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = leader (issues the MMAs), 1 = peer
    const int item0 = p.run[p.first_run].begin;
    const int nitems = p.run[p.end_run].begin - item0;
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
        for (int g = 0; g < EPI_GROUPS; ++g)
            for (int s = 0; s < PUB_DEPTH; ++s) {
                mbar_init(&mbox.full[g][s], 1);
                mbar_init(&mbox.empty[g][s], 1);
            }
        for (int s = 0; s < SDEPTH; ++s) {
            mbar_init(&sring.full[s], 1);
            mbar_init(&sring.empty[s], SCONSUMERS);
            mbar_init(&sring.taken[s], 1);
        }
        mbar_init(&mma_done_bar, 1);
        fence_mbar_init();
        aborted = 0;
    }
    if (threadIdx.x == 32) {
        for (int i = 0; i < p.nbanks; ++i)
            for (int k = 0; k < TM_COUNT; ++k)
                if (k != TM_OUT || p.bank[i].out_tma) tma_prefetch_desc(&p.bank[i].tm[k]);
    }
    if (warp == 1) tmem_alloc_pair(&tmem_slot, TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    pdl_wait_previous();  // everything above overlapped the previous kernel's tail
    const uint32_t tmem = tmem_slot;
    int issued = 0;      // producer: k-blocks whose loads were armed (in the whole CTA life)
    int epi_tiles = 0;   // epilogue group: tiles whose input loads were armed

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int it = 0;
            for (int k = 0;; ++k) {
                const Work w = sched_take(sring, k, p.err);
                if (w.t() == 0x7fffffff) aborted = 1;
                if (rank == 0) mbar_arrive_relaxed(&sring.taken[k % SDEPTH]);
                if (w.t() >= nitems) break;
                // the scheduler saw the item's inputs complete (acquire); these TMA reads follow
                asm volatile("fence.proxy.async.global;" ::: "memory");
                const int nkb = w.nkb();
                bool ok = true;
#ifdef ANVIL_TIMELINE
                unsigned long long tl_wait = 0;
#endif
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t r = static_cast<uint32_t>(it / STAGES);
#ifdef ANVIL_TIMELINE
                    const unsigned long long tl_c0 = clock64();
#endif
                    if (!mbar_wait(&empty_bar[s], (r & 1u) ^ 1u, p.err)) {
                        ok = false;
                        break;
                    }
#ifdef ANVIL_TIMELINE
                    tl_wait += clock64() - tl_c0;
                    if (kb == nkb - 1 && rank == 0) TL_PUT(w.t(), TL_PROD_WAIT_CLK, tl_wait);
#endif
                    if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], w.shared_ab() ? 2 * A_STAGE : 2 * STAGE);
                    if (kb == 0 && rank == 0) TL_PUT(w.t(), TL_PROD_FIRST, globaltimer_ns());
                    load_kblock(p, w, kb, rank, smem + s * STAGE, map_to_rank(&full_bar[s], 0));
                    issued = it + 1;
                }
                if (!ok) {
                    aborted = 1;
                    break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (leader CTA)
            // The issuing thread is the k-loop's critical path: between two k-blocks it has
            // only the time the queued MMAs take, so the next stage's barrier is tested
            // (without blocking) while this k-block's MMAs run, and a blocking wait happens
            // only when that test found the stage not yet loaded.
            const uint32_t stage0 = smem_u32(smem);
            int s = 0, mt = 0;
            uint32_t ph = 0;     // parity of stage s's next fill
            bool ready = false;  // that fill already seen complete
            for (int lt = 0;; ++lt) {
                const Work w = sched_take(sring, lt, p.err);
                if (w.t() == 0x7fffffff) aborted = 1;
                if (w.t() >= nitems) break;
                const bool xu = op_xupdate(w.op());
                const int nkb = w.nkb();
                const bool shared_ab = w.shared_ab();
                // operands staged MN-major: Y in the X-update, and the k-blocks left of a
                // symmetric operand's diagonal block, read from the transposed upper block (as
                // the producer loaded them)
                const int kb_a_mn = w.map(1) >= 0 ? w.bi() * (PAIR / BK) : 0;
                const int kb_b_mn = xu ? nkb : (w.map(3) >= 0 ? w.bj() * (PAIR / BK) : 0);
                const int ab = mt & 1;
                const uint32_t u = static_cast<uint32_t>(mt >> 1);
                ++mt;
                TL_PUT(w.t(), TL_MMA_TAKEN, globaltimer_ns());
                if (!mbar_wait(&tempty_bar[ab], (u & 1u) ^ 1u, p.err)) {
                    aborted = 1;
                    break;
                }
                TL_PUT(w.t(), TL_MMA_ACC_FREE, globaltimer_ns());
                tc_fence_after();
                const uint32_t dacc = tmem + static_cast<uint32_t>(ab * BN);
                bool ok = true;
#ifdef ANVIL_TIMELINE
                unsigned long long tl_wait = 0;
#endif
                for (int kb = 0; kb < nkb; ++kb) {
#ifdef ANVIL_TIMELINE
                    const unsigned long long tl_c0 = clock64();
#endif
                    if (!ready && !mbar_wait(&full_bar[s], ph, p.err)) {
                        ok = false;
                        break;
                    }
#ifdef ANVIL_TIMELINE
                    if (kb > 0) tl_wait += clock64() - tl_c0;  // waits inside the k-loop only
                    if (kb == nkb - 1) TL_PUT(w.t(), TL_MMA_WAIT_CLK, tl_wait);
#endif
                    if (kb == 0) {
                        TL_PUT(w.t(), TL_MMA_FIRST, globaltimer_ns());
                        TL_PUT(w.t(), TL_MMA_FIRST_CLK, clock64());
                    }
                    tc_fence_after();
                    const uint32_t a0 = stage0 + static_cast<uint32_t>(s * STAGE);
                    const uint32_t b0 = shared_ab ? a0 : a0 + A_STAGE;
                    const bool a_mn = kb < kb_a_mn, b_mn = kb < kb_b_mn;
                    const uint32_t idesc = idesc_bf16_f32(PAIR, PAIR, a_mn, b_mn);
                    // K-major: a 16-deep k-step is 32 bytes along the row; MN-major: 64-element
                    // chunks 8 KB apart, a k-step is 16 rows of 128 bytes
                    const uint32_t a_lo = sw128_desc_lo(a0, a_mn ? 8192 : 16);
                    const uint32_t b_lo = sw128_desc_lo(b0, b_mn ? 8192 : 16);
                    const uint32_t a_step = a_mn ? 2048 >> 4 : 32 >> 4, b_step = b_mn ? 2048 >> 4 : 32 >> 4;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(dacc, sw128_desc(a_lo + kk * a_step), sw128_desc(b_lo + kk * b_step), idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    const int s_next = s + 1 == STAGES ? 0 : s + 1;
                    const uint32_t ph_next = s_next == 0 ? ph ^ 1u : ph;
                    ready = mbar_test_wait(smem_u32(&full_bar[s_next]), ph_next);
                    umma_commit_pair(&empty_bar[s], 3);  // frees stage s in both CTAs
                    if (kb == nkb - 1) {
                        TL_PUT(w.t(), TL_MMA_LAST, globaltimer_ns());
                        TL_PUT(w.t(), TL_MMA_LAST_CLK, clock64());
                    }
                    s = s_next;
                    ph = ph_next;
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
    } else if (warp == SCHED_WARP) {
        if (lane == 0 && rank == 0) {
            // ---------------- scheduler (leader CTA)
            for (int k = 0;; ++k) {
                // take a pair's next item only once its producer has started the one SAHEAD
                // entries before: an item taken much earlier would wait behind this pair's work
                if (k >= SAHEAD &&
                    !mbar_wait(&sring.taken[(k - SAHEAD) % SDEPTH], ((k - SAHEAD) / SDEPTH) & 1, p.err)) {
                    aborted = 1;
                    break;
                }
                const unsigned next = aborted ? static_cast<unsigned>(nitems) : atomicAdd(p.next_item, 1u);
                int t = next >= static_cast<unsigned>(nitems) ? nitems : static_cast<int>(next);
                Work w = make_work(p, item0, nitems, t);
                if (t < nitems) {
                    TL_PUT(t, TL_META, (static_cast<unsigned long long>(blockIdx.x >> 1)) |
                                           (static_cast<unsigned long long>(w.w0.y) << 16) |
                                           (static_cast<unsigned long long>(w.mat()) << 48));
                    TL_PUT(t, TL_TILE, static_cast<unsigned long long>(w.bi()) |
                                           (static_cast<unsigned long long>(w.bj()) << 16) |
                                           (static_cast<unsigned long long>(w.nkb()) << 32));
                    TL_PUT(t, TL_SCHED_TAKE, globaltimer_ns());
                }
                // the entry goes out once the phases the item reads are complete for its
                // matrix, so no role of the pair waits on another pair after taking it
                if (t < nitems && !deps_wait(p, work_item(w))) {
                    aborted = 1;
                    t = nitems;
                    w = make_work(p, item0, nitems, t);
                }
                if (t < nitems) TL_PUT(t, TL_SCHED_READY, globaltimer_ns());
                if (!sched_push(sring, k, w, p.err)) {
                    aborted = 1;
                    break;
                }
                if (t < nitems) TL_PUT(t, TL_SCHED_PUSH, globaltimer_ns());
                if (t >= nitems) break;
            }
        }
    } else if (warp == PUB_WARP) {
        if (lane == 0) {
            // ---------------- publisher: one release add per finished tile and group
            int k[EPI_GROUPS] = {0, 0};
            int open = EPI_GROUPS;
            unsigned long long t0 = globaltimer_ns();
            while (open > 0) {
                bool got = false;
                for (int g = 0; g < EPI_GROUPS; ++g) {
                    if (k[g] < 0) continue;
                    const int s = k[g] % PUB_DEPTH;
                    if (!mbar_test_wait(smem_u32(&mbox.full[g][s]), (k[g] / PUB_DEPTH) & 1)) continue;
                    unsigned* cnt = mbox.slot[g][s];
                    if (cnt) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
                    mbar_arrive_cta(&mbox.empty[g][s]);
                    k[g] = cnt ? k[g] + 1 : -1;
                    if (!cnt) --open;
                    got = true;
                }
                if (got) {
                    t0 = globaltimer_ns();
                } else {
                    __nanosleep(128);
                    if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                        atomicOr(p.err, DEVERR_TIMEOUT);
                        aborted = 1;
                        break;
                    }
                }
            }
        }
    } else {
        // ---------------- epilogue: warps 2-9, TMEM lane quadrant = warp % 4
        const int quad = warp & 3;
        EpiCtx x;
        x.stg = smem + STAGES * STAGE;  // staging boxes (1024-aligned)
        x.epi_bar = epi_bar;
        x.r = quad * 32 + lane;
        x.grp = (warp - 2) >> 2;
        x.lane = lane;
        x.leader = ((warp - 2) & 3) == 0 && lane == 0;
        x.last_box = -1;
        x.fail = false;
        x.npub = 0;
        const uint32_t tempty_leader0 = map_to_rank(&tempty_bar[0], 0);
        const uint32_t tempty_leader1 = map_to_rank(&tempty_bar[1], 0);
        int mt = 0;
        bool pending = false;  // the group's latest tile, published after the next one
        Item pend = {0, 0, 0, 0, 0};
        for (int lt = 0;; ++lt) {
            if (x.leader) {
                // the group's next item; a wait that may be long never holds back this
                // group's last tile
                if (pending && !mbar_test_wait(smem_u32(&sring.full[lt % SDEPTH]), (lt / SDEPTH) & 1)) {
                    bulk_wait_all();
                    send_done(mbox, x, tile_counter(p, pend), p.err);
                    pending = false;
                }
                const Work wn = sched_take(sring, lt, p.err);
                if (wn.t() == 0x7fffffff) x.fail = true;
                grp_work[x.grp][lt & 1][0] = wn.w0;
                grp_work[x.grp][lt & 1][1] = wn.w1;
            }
            // the group stops together: at its last item, or once any wait of any role
            // (or of any thread of the group) gave up
            if (named_barrier_or(1 + x.grp, 128, x.fail || aborted)) {
                aborted = 1;
                break;
            }
            Work w;
            w.w0 = grp_work[x.grp][lt & 1][0];
            w.w1 = grp_work[x.grp][lt & 1][1];
            if (w.t() >= nitems) break;
            const Item c = work_item(w);
            const CascadePhase& P = p.phase[c.ph];
            const CascadeBank& bk = p.bank[c.bank];
            const int op = w.op();
            const uint32_t in_phase = static_cast<uint32_t>(epi_tiles) & 1u;
            if (!op_gram(op)) {
                // the group's quarters of the tile's input, once the group's earlier TMA
                // stores have finished reading the boxes
                if (x.leader) {
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    bulk_wait_read_all();
                    for (int q = 2 * x.grp; q < 2 * x.grp + 2; ++q) {
                        mbar_arrive_expect_tx(&epi_bar[q], QBOX);
                        tma_load_3d(x.stg + q * QBOX, &bk.tm[P.map_in], &epi_bar[q],
                                    c.bj * PAIR + 64 * q, c.bi * PAIR + TILE * static_cast<int>(rank), c.mat);
                    }
                }
                ++epi_tiles;
                x.last_box = -1;  // every box of the group is now an input box
            }
            const int ab = mt & 1;
            const uint32_t u = static_cast<uint32_t>(mt >> 1);
            ++mt;
            if (!mbar_wait(&tfull_bar[ab], u & 1u, p.err)) x.fail = true;
            if (x.leader && x.grp == 0 && rank == 0) TL_PUT(w.t(), TL_EPI_START, globaltimer_ns());
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(ab * BN);
            const uint32_t tempty = ab ? tempty_leader1 : tempty_leader0;
            switch (op) {
                case OP_GRAM: epi_tile<OP_GRAM>(p, bk, P, c, rank, x, tbase, tempty, in_phase); break;
                case OP_GRAM_NORM: epi_tile<OP_GRAM_NORM>(p, bk, P, c, rank, x, tbase, tempty, in_phase); break;
                case OP_SQPOLY: epi_tile<OP_SQPOLY>(p, bk, P, c, rank, x, tbase, tempty, in_phase); break;
                case OP_XUPDATE: epi_tile<OP_XUPDATE>(p, bk, P, c, rank, x, tbase, tempty, in_phase); break;
                default: epi_tile<OP_XUPDATE_OUT>(p, bk, P, c, rank, x, tbase, tempty, in_phase); break;
            }
            if (x.leader && x.grp == 0 && rank == 0) TL_PUT(w.t(), TL_EPI_END, globaltimer_ns());
            // publish the group's previous tile: its stores are older than this tile's two
            // (one per quarter), so they have long completed
            if (x.leader && pending) {
                if (op != OP_XUPDATE_OUT || bk.out_tma) bulk_wait_all_but_two();
                else bulk_wait_all();
                send_done(mbox, x, tile_counter(p, pend), p.err);
            }
            pending = true;
            pend = c;
        }
        if (x.leader) {
            bulk_wait_all();  // every store of this group has completed
            if (pending && !aborted) send_done(mbox, x, tile_counter(p, pend), p.err);
            send_done(mbox, x, nullptr, p.err);  // the group's last message
            if (aborted && epi_tiles > 0)  // and every input load it armed has landed
                for (int q = 2 * x.grp; q < 2 * x.grp + 2; ++q)
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
    if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

static int g_max_pairs[64];  // co-resident CTA pairs per device (0 = unknown)

cudaError_t launch_cascade(const CascadeParams& p, cudaStream_t stream) {
    const int nitems = p.run[p.end_run].begin - p.run[p.first_run].begin;
    if (nitems <= 0) return cudaSuccess;
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
    cfg.dynamicSmemBytes = GEMM_SMEM;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int& maxp = g_max_pairs[dev & 63];
    if (maxp == 0) {
        cfg.gridDim = dim3(2 * (p.sm_count / 2), 1, 1);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, cascade_kernel, &cfg);
        if (e) return e;
        maxp = clusters > 0 ? clusters : 1;
    }
    // no more pairs than can be resident at once: items wait on other pairs' items
    const int pairs = nitems < maxp ? nitems : maxp;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, cascade_kernel, p);
}

cudaError_t timeline_copy(void* host, size_t bytes, int clear) {
#ifdef ANVIL_TIMELINE
    void* dev = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&dev, g_timeline);
    if (e) return e;
    if (host && bytes) {
        const size_t n = bytes < sizeof(g_timeline) ? bytes : sizeof(g_timeline);
        if ((e = cudaMemcpy(host, dev, n, cudaMemcpyDeviceToHost))) return e;
    }
    return clear ? cudaMemset(dev, 0, sizeof(g_timeline)) : cudaSuccess;
#else
    (void)host;
    (void)bytes;
    (void)clear;
    return cudaErrorNotSupported;
#endif
}

cudaError_t gemm_prepare() {
    return cudaFuncSetAttribute(cascade_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
}

}  // namespace anvil
