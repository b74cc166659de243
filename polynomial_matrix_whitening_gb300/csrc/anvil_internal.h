// anvil_internal.h -- kernel parameter blocks and launchers shared by libanvil's
// translation units (not part of the public ABI).
//
// Working layout.  Every matrix is carried in small-side-major form Y [s_pad, L_pad]
// (s = min(m, n) rows, L = max(m, n) columns, row-major, bf16): Y = X for a wide
// matrix (m <= n) and Y = X^T for a tall one.  Both branches of the page's cascade
// are then the same three products,
//     A = Y Y^T,   B = b A + c A A,   Y <- a Y + B Y,
// because for a tall X, X^T X = Y Y^T and (a X + X B)^T = a Y + B Y (B is symmetric).
// s_pad and L_pad round s and L up to 256; the padding is zero and
// stays zero through every step (zero rows and columns of Y give zero rows and
// columns of A and B), so it changes no result.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace anvil {

constexpr int TILE = 128;            // GEMM rows per CTA
constexpr int PAIR = 256;            // GEMM tile edge per CTA pair, and the padding unit
constexpr int LPAD = 256;            // padding unit of the long side
constexpr int BK = 64;               // GEMM k-block: one 128-byte swizzle row of bf16
constexpr int LBLK = 64;             // momentum-kernel tile edge; one diagonal partial each
constexpr int MAX_BANKS = 8;         // banks per call

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Launches `kernel` with programmatic stream serialisation: its prologue may overlap the
// tail of the previous kernel on the stream; the kernel calls pdl_wait_previous() before
// touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The step-to-tail link buffer of one bank (anvil_tail_link_bytes): the slow rail's sign
// words, uint64 [g, nck, m, 2] for 64-column chunk k, out row r: word 0 bit 16 q + t is
// the sign of the slow rail at column 64 k + 4 t + q (t < 16, q < 4), word 1's same bit
// says that the value is zero, below 2^-100 in magnitude, infinite or NaN (the tail then
// reads the fp32 rail itself).
struct LinkLayout {
    int nck;
    size_t total;
};
inline LinkLayout link_layout(int g, int m, int n) {
    LinkLayout k;
    k.nck = (n + 63) / 64;
    k.total = (16 * static_cast<size_t>(g) * m * k.nck + 255) & ~static_cast<size_t>(255);
    return k;
}

// Bits of the device error word (set with atomicOr, read by anvil_device_error).
enum : unsigned { DEVERR_TIMEOUT = 1u, DEVERR_BOUNDS = 2u };

// ---------------------------------------------------------------- momentum + cast
struct MomentumBank {
    const void* grad;    // fp32, or bf16 bits when grad_bf16   // [g, m, n]
    float* velocity;     // [2, g, m, n]
    uint16_t* y;         // Y_raw [g, s_pad, L_pad]
    float* part;         // [g, nlb, s_pad]: sums of squares of the bf16 values per 64-block
    int g, m, n, tall, s_pad, L_pad, nlb;
    int tiles_r, tiles_c;  // 64x64 tiles over the padded natural extent [rows, cols]
    uint64_t* gate;        // tail link: slow-rail sign words [g, nck, m, 2] (NULL: none)
    int nck;               // 64-column chunks per row, (n + 63) / 64
    int tile_begin;        // first tile of this bank in the grouped grid
    int vec4;              // n % 4 == 0 and aligned grad/velocity: 4-element vector path
    int grad_bf16;
    float momentum, fast_beta, fast_weight, slow_beta;
};
struct MomentumParams {
    MomentumBank bank[MAX_BANKS];
    int nbanks, total_tiles;
    const float* dev_scalars;  // [nbanks][4] on the device, or null
    unsigned* err;
};
cudaError_t launch_momentum(const MomentumParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- d and normalisation
struct NormBank {
    const float* part;  // [g, nlb, s_pad]
    int g, s_pad, L_pad, nlb;
    int mat_begin;      // first matrix of this bank among all matrices of the call
};
struct NormParams {
    NormBank bank[MAX_BANKS];
    int nbanks, total_mats;
    float margin, eps;
    float* d;  // [total_mats]
    unsigned* counters;  // [total_mats + SCHED_COUNTERS] cascade counters, zeroed by norm_d
    unsigned* err;
};
// d[mat] = sqrt(sum_i float(bf16(sum of the partials of i))) * margin + eps; also zeroes
// the matrix's cascade completion counters.
cudaError_t launch_norm_d(const NormParams& p, cudaStream_t stream);

// The normalisation X / d: Y1 = bf16(Y0 / d[mat]) over the padded extent [s_pad, L_pad]
// of every matrix, in 8-element (16-byte) chunks.  A block converts NX_BLOCK_CHUNKS
// consecutive chunks of one matrix (s_pad and L_pad are multiples of 256, so a matrix is
// a whole number of blocks); the blocks are numbered bank by bank.
constexpr int NX_BLOCK_CHUNKS = 1024;
static_assert((PAIR * LPAD / 8) % NX_BLOCK_CHUNKS == 0, "a padded matrix is a whole number of X / d blocks");
struct NormXBank {
    const uint16_t* y0;   // [g, s_pad, L_pad] X_raw
    uint16_t* y1;         // [g, s_pad, L_pad] X / d
    const float* d;       // [g]
    int block_begin;      // first block of this bank
    int blocks_per_mat;   // s_pad * L_pad / 8 / NX_BLOCK_CHUNKS
};
struct NormXParams {
    NormXBank bank[MAX_BANKS];
    int nbanks;
    int total_blocks;
};
cudaError_t launch_normalize(const NormXParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- the cascade kernel
// One persistent tcgen05 kernel walks every phase of the cascade (anvil_gemm.cu).
enum PhaseOp : int {
    OP_GRAM = 0,        // A = bf16(Y Y^T)                    (diagonal and upper 256-blocks)
    OP_GRAM_NORM = 1,   // A = bf16(bf16(Y Y^T) / d^2)        (the first Gram, on X_raw)
    OP_SQPOLY = 2,      // B = bf16(b A + c A A)              (diagonal and upper 256-blocks)
    OP_XUPDATE = 3,     // Y' = bf16(a Y + B Y)
    OP_XUPDATE_OUT = 4  // the same, written to out in the natural [m, n] layout
};

// Tensor maps of one bank (3-D bf16 over [g][rows][cols]).
enum MapSlot : int {
    TM_YK0 = 0,  // Y0, box {64, 128}, 128-byte swizzle: K-major operand, epilogue boxes
    TM_YK1 = 1,  // Y1, the same
    TM_YN0 = 2,  // Y0, box {64, 64}: MN-major operand of the X-update
    TM_YN1 = 3,  // Y1, the same
    TM_A = 4,    // A [g][s_pad][s_pad], box {64, 128}
    TM_B = 5,    // B, the same
    TM_OUT = 6,  // out [g][m][n], box {64, 128} (wide) or {64, 64} (tall), rows 16-byte aligned
    TM_AN = 7,   // A, box {64, 64}: an upper block read as the transpose of a lower one
    TM_BN = 8,   // B, the same
    TM_COUNT = 9
};

constexpr int MAX_CASCADE_MAPS = 16;                      // spectral maps per call
constexpr int MAX_PHASES = 3 * MAX_CASCADE_MAPS;          // GRAM_NORM, then 3 per map but the first map's Gram

struct CascadeBank {
    CUtensorMap tm[TM_COUNT];
    uint16_t* a;        // A [g, s_pad, s_pad]
    uint16_t* b;        // B [g, s_pad, s_pad]
    uint16_t* out;      // out [g, m, n]
    const uint16_t* y0; // X_raw [g, s_pad, L_pad] (the first Gram's operand)
    uint16_t* y1;       // normalised X (the first X-update's input)
    const float* d;     // [g] normaliser of this bank's matrices
    int g, s_pad, L_pad, m, n, tall;
    int out_tma;        // out is written through TM_OUT (rows 16-byte aligned; tall: transposed boxes)
    int T, ntl;         // s_pad / PAIR and L_pad / PAIR: row and column blocks of Y
    int mat_begin;      // first matrix of this bank among all matrices of the call
};

// A phase: one op of the cascade (over every matrix of every bank).  A = Y Y^T and B are
// symmetric; the kernel writes their diagonal and upper 256x256 blocks only.
struct CascadePhase {
    int op;
    int map_a, map_b, map_in, map_out;  // MapSlot of each operand (-1: none)
    // A and B are stored as their upper-triangle 256-blocks only: a k-block of a product
    // operand that falls below the diagonal is read, MN-major, from the transposed upper
    // block through these maps (-1: the operand is not symmetric)
    int map_a_t, map_b_t;
    float a, b, c;                      // the map's coefficients
    // before an item of matrix i of bank q loads anything: chain[i] >= need_chain[q]
    // (0: no wait)
    unsigned need_chain[MAX_BANKS];
};

// The order in which the kernel walks its items: a list of runs, each the tiles of one
// phase for a range of matrices of one bank (matrix by matrix, block row by block row),
// numbered from `begin`.  Any order is valid in which every phase of a matrix comes after
// the phases it reads.
struct CascadeRun {
    int begin;        // first item (global index) of the run
    uint8_t phase;
    uint8_t bank;
    uint16_t mat0;    // first matrix (within the bank)
    uint32_t nmat;    // matrices in the run
};
constexpr int MAX_RUNS = MAX_PHASES * MAX_BANKS;  // phase by phase, one run per bank

struct CascadeParams {
    CascadeBank bank[MAX_BANKS];
    CascadePhase phase[MAX_PHASES];
    CascadeRun run[MAX_RUNS + 1];  // run[nruns].begin = the item count
    int nbanks, nphases, nruns;
    int first_run, end_run;  // this launch walks runs [first_run, end_run)
    int sm_count;
    // Completion counters per matrix, zeroed by norm_d_kernel each step: every finished
    // tile adds one per epilogue warp group per CTA (4 per tile) to chain[] (the chain of
    // product phases, each of which waits for the one before it).
    unsigned* chain;
    // this launch's item counter (zeroed by norm_d_kernel each step): every CTA pair takes
    // its next item with an atomic add
    unsigned* next_item;
    unsigned* err;
};
constexpr unsigned SIGNALS_PER_TILE = 4;
// item counters per step: one for the fused launch, one per phase for traced steps
constexpr int SCHED_COUNTERS = MAX_PHASES + 1;
cudaError_t launch_cascade(const CascadeParams& p, cudaStream_t stream);
cudaError_t gemm_prepare();  // sets the cascade kernel's shared-memory limit on this device

// Per-item timeline of the cascade kernel (a library built with -DANVIL_TIMELINE): the
// 64-bit fields each item of the latest launches records.  timeline_copy copies up to
// `bytes` to the host (if host != NULL), then zeroes the buffer if `clear`;
// cudaErrorNotSupported in a library built without it.
constexpr int TL_ITEMS = 16384;  // ANVIL_TIMELINE_ITEMS
enum TimelineField : int {
    TL_META = 0,          // pair | (op | bank << 8 | phase << 16) << 16 | matrix << 48
    TL_TILE = 1,          // block row | block column << 16 | k-blocks << 32
    TL_SCHED_TAKE = 2,    // scheduler took the item (ns)
    TL_SCHED_READY = 3,   // its input phases were complete (ns)
    TL_SCHED_PUSH = 4,    // its entry was in the ring (ns)
    TL_PROD_FIRST = 5,    // producer armed its first k-block (ns)
    TL_MMA_TAKEN = 6,     // MMA issuer read the entry (ns)
    TL_MMA_ACC_FREE = 7,  // its accumulator was free (ns)
    TL_MMA_FIRST = 8,     // first k-block landed, first MMA issued (ns)
    TL_MMA_LAST = 9,      // last k-block's MMAs issued (ns)
    TL_EPI_START = 10,    // epilogue found the accumulator complete (ns)
    TL_EPI_END = 11,      // epilogue done with the tile (ns)
    TL_MMA_FIRST_CLK = 12,
    TL_MMA_LAST_CLK = 13,
    TL_MMA_WAIT_CLK = 14,   // SM cycles the MMA issuer waited for k-blocks 1.. to land
    TL_PROD_WAIT_CLK = 15,  // SM cycles the producer waited for free ring stages
    TL_FIELDS = 16
};
cudaError_t timeline_copy(void* host, size_t bytes, int clear);

// ---------------------------------------------------------------- tracing / self-test
// dst [g, m, n] (natural layout) <- Y [g, s_pad, L_pad] (small-side-major), bf16.
cudaError_t launch_extract_x(const uint16_t* y, uint16_t* dst, int g, int m, int n, int tall,
                             int s_pad, int L_pad, cudaStream_t stream);
// dst [g, s, s] <- src [g, s_pad, s_pad], bf16, from the diagonal and upper 256-blocks of a
// symmetric src (a lower block is the transpose of the upper one).
cudaError_t launch_extract_sq(const uint16_t* src, uint16_t* dst, int g, int s, int s_pad,
                              cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned timeout_us, unsigned* err, cudaStream_t stream);


// Device address of the current device's error word (null if it cannot be had).
unsigned* device_error_word();
// Reads the error word (and clears it if asked) after the work queued on `stream`, with one
// atomic on the device; waits for that stream only.
cudaError_t read_error_word_on_stream(unsigned* err, int clear, unsigned* word, cudaStream_t stream);

}  // namespace anvil
