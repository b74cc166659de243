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
constexpr int MAX_LAUNCH_BANKS = 4;  // banks grouped into one GEMM launch

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
    const uint16_t* y;  // X_raw [g, s_pad, L_pad]
    uint16_t* y_out;    // normalised X [g, s_pad, L_pad]
    const float* part;  // [g, nlb, s_pad]
    int g, s_pad, L_pad, nlb;
    int mat_begin;      // first matrix of this bank among all matrices of the call
    long long vec_begin;  // first 8-element vector of this bank in the grouped grid
};
struct NormParams {
    NormBank bank[MAX_BANKS];
    int nbanks, total_mats;
    long long total_vecs;
    float margin, eps;
    float* d;  // [total_mats]
    unsigned* err;
};
// d[mat] = sqrt(sum_i float(bf16(sum of the partials of i))) * margin + eps.
cudaError_t launch_norm_d(const NormParams& p, cudaStream_t stream);
// Y_out <- bf16(float(Y) / d[mat]) over every bank.
cudaError_t launch_normalize(const NormParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05 GEMMs
enum GemmOp : int {
    OP_GRAM = 0,        // A = bf16(Y Y^T)                    (upper tiles, mirrored)
    OP_GRAM_NORM = 1,   // A = bf16(bf16(Y Y^T) / d^2)        (the first Gram)
    OP_SQPOLY = 2,      // B = bf16(b A + c A A)              (upper tiles, mirrored)
    OP_XUPDATE = 3,     // Y' = bf16(a Y + B Y)
    OP_XUPDATE_OUT = 4  // the same, written to out in the natural [m, n] layout
};

struct GemmBank {
    CUtensorMap tm_a;     // A operand, K-major, box {64, 128, 1}
    CUtensorMap tm_b;     // B operand: K-major box {64, 128, 1}, or (xupdate) MN-major {64, 64, 1}
    CUtensorMap tm_c;     // epilogue input (A for sqpoly, Y for xupdate), box {64, 128, 1}
    CUtensorMap tm_d;     // epilogue output, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tm_e;     // transposed epilogue output (mirror tile / tall out), box {128, 64, 1}
    const uint16_t* src;  // epilogue input: A (sqpoly) or Y (xupdate)
    uint16_t* dst;        // output
    const float* d;       // [g] normaliser of this bank's matrices (gram_norm)
    int g, s_pad, L_pad, m, n, tall;
    int out_tma;          // xupdate_out: `out` rows are 16-byte aligned (TMA stores)
    int T;                // s_pad / PAIR (row blocks)
    int nt_n;             // column blocks (T for sym ops, L_pad / PAIR for xupdate)
    int tiles_per_mat;
    int tile_begin;
    int num_kb;           // k-blocks of BK
};
struct GemmParams {
    GemmBank bank[MAX_LAUNCH_BANKS];
    int nbanks, total_tiles;
    int sm_count;  // persistent grid: CTA pairs up to the co-resident limit
    float a, b, c;
    unsigned* err;
};
cudaError_t launch_gemm(GemmOp op, const GemmParams& p, cudaStream_t stream);
int gemm_tile_cols(GemmOp op);  // output tile columns of this op's kernel
cudaError_t gemm_prepare();  // sets the GEMM kernels' shared-memory limit on this device

// ---------------------------------------------------------------- tracing / self-test
// dst [g, m, n] (natural layout) <- Y [g, s_pad, L_pad] (small-side-major), bf16.
cudaError_t launch_extract_x(const uint16_t* y, uint16_t* dst, int g, int m, int n, int tall,
                             int s_pad, int L_pad, cudaStream_t stream);
// dst [g, s, s] <- src [g, s_pad, s_pad], bf16.
cudaError_t launch_extract_sq(const uint16_t* src, uint16_t* dst, int g, int s, int s_pad,
                              cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned timeout_us, unsigned* err, cudaStream_t stream);


// Device address of the current device's error word (null if it cannot be had).
unsigned* device_error_word();

}  // namespace anvil
