/*
 * anvil.h -- C ABI of libanvil, the ANVIL bank step on GB300 (sm_103a).
 *
 * The operation is the one defined on the page "modded-nanogpt
 * track_1_short/optim/anvil.py", function `anvil_cascade` and the constants
 * above it (ANVIL_MAPS, RAIL_FAST_BETA / RAIL_SLOW_BETA / RAIL_FAST_WEIGHT,
 * FROBENIUS_MARGIN / FROBENIUS_EPS).  For every matrix G of a bank [g, m, n]:
 *
 *   v0 <- v0 + (1 - fast_beta) (G - v0)          fast rail   (velocity[0])
 *   v1 <- v1 + (1 - slow_beta) (G - v1)          slow rail   (velocity[1])
 *   blend = w v0 + (1 - w) v1                    w = fast_weight
 *   X  = bf16(G + momentum (blend - G))          Nesterov lookahead
 *   tall (m > n): A = X^T X, update X <- a X + X B
 *   wide (m <= n, square included): A = X X^T, update X <- a X + B X
 *   d  = sqrt(trace of the bf16 first Gram) * margin + eps
 *   X  <- bf16(X / d), A <- bf16(A / d^2)
 *   for each map (a, b, c): [A = bf16(Gram(X)) after the first]
 *       B = bf16(b A + c A A);  X <- bf16(a X + X B  |  a X + B X)
 *   out = X
 *
 * Every number is computed on the GPU by this library's own kernels; there is
 * no CPU path.  All calls are asynchronous on the given stream (a
 * cudaStream_t / CUstream handle passed as void*; NULL = legacy default
 * stream).  A step is four kernels on that stream: momentum + cast, the normaliser d,
 * the normalisation X / d, and one persistent kernel for every product of every map.
 * No call below allocates, frees or synchronises, except anvil_bank_step on its first
 * use of a size (documented there), the error reads anvil_last_device_error (waits for
 * its stream) and anvil_device_error (waits for the device).  Errors are returned as
 * status codes; no exception crosses the ABI.
 */
#ifndef ANVIL_H
#define ANVIL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ANVIL_OK = 0,
    ANVIL_ERR_INVALID_ARG = 1,       /* null pointer, g/m/n < 1, nmaps out of range, ... */
    ANVIL_ERR_UNSUPPORTED_SHAPE = 2, /* a dimension above ANVIL_MAX_DIM / ANVIL_MAX_BATCH, or a
                                        call of over 2^40 padded elements (terabytes of workspace) */
    ANVIL_ERR_ALIGNMENT = 3,         /* pointer not aligned to its element size / workspace to 256 B */
    ANVIL_ERR_ALIAS = 4,             /* a written buffer overlaps another buffer of the call */
    ANVIL_ERR_WORKSPACE = 5,         /* workspace too small, or cannot be allocated during capture */
    ANVIL_ERR_CUDA = 6,              /* a CUDA runtime/driver call or a launch failed */
    ANVIL_ERR_TIMEOUT = 7,           /* a bounded device-side wait gave up (see anvil_last_device_error) */
    ANVIL_ERR_DEVICE = 8,            /* current device is not sm_103 (the kernels are sm_103a only) */
    ANVIL_ERR_UNAVAILABLE = 9        /* a diagnostic this build of the library does not include */
} anvil_status;

/* One quintic spectral map f(s) = a s + b s^3 + c s^5 (an ANVIL_MAPS entry). */
typedef struct { float a, b, c; } anvil_map;

/* Per-step scalars of one bank (the page's AnvilBank momentum / fast_beta /
 * fast_weight, plus the slow rail's beta, RAIL_SLOW_BETA there). */
typedef struct { float momentum, fast_beta, fast_weight, slow_beta; } anvil_scalars;

/* One bank of g matrices of m x n.  All pointers are DEVICE pointers, row-major,
 * caller-owned:
 *   grad      [g, m, n]    fp32, or bf16 bits when grad_bf16 != 0 (the page's bank
 *                          gradient is bf16); read only (never written)
 *   velocity  [2, g, m, n] fp32, read and written in place; rail 0 fast, rail 1 slow
 *   out       [g, m, n]    bf16 bits, written
 *   tail_link  optional DEVICE buffer of anvil_tail_link_bytes(g, m, n) bytes, 256-byte
 *              aligned, or NULL: the step also writes there the sign of every slow-rail
 *              value (2 bits per element: the sign, and whether the tail must read the
 *              value itself), so that anvil_update_tail given the same buffer gates its
 *              decay without reading the fp32 slow rail (0.25 instead of 4 bytes per element)
 * grad must be aligned to its element size, velocity to 4 bytes, out to 2 bytes; out
 * and tail_link must not overlap grad, velocity or any buffer of another bank in the
 * same call.  `scalars` is used when the call's device scalar array is NULL. */
typedef struct {
    const void* grad;
    float* velocity;
    uint16_t* out;
    int g, m, n;
    anvil_scalars scalars;
    int grad_bf16;
    void* tail_link;
} anvil_bank_desc;

/* Bytes of the step-to-tail link buffer of one bank of g matrices of m x n (0 if the
 * shape is invalid).  Its contents are internal to the library: written by the step
 * (anvil_multi_bank_step, anvil_bank_step_traced), read by anvil_update_tail, valid
 * until the bank's next step. */
size_t anvil_tail_link_bytes(int g, int m, int n);

#define ANVIL_MAX_MAPS 16     /* maps per call */
#define ANVIL_MAX_BANKS 8     /* banks per anvil_multi_bank_step call */
#define ANVIL_MAX_DIM 16384   /* largest m or n */
#define ANVIL_MAX_BATCH 65535 /* largest g */

/* Writes the page's six ANVIL_MAPS into maps[0..5] (if cap >= 6) and returns 6. */
int anvil_default_maps(anvil_map* maps, int cap);

/* Bytes of device workspace anvil_multi_bank_step needs for these banks
 * (0 if the descriptors are invalid).  Depends only on g, m, n of each bank. */
size_t anvil_workspace_bytes(const anvil_bank_desc* banks, int nbanks);

/* One ANVIL step over nbanks banks, every kernel grouped across the banks.
 *   banks      host array of nbanks descriptors (1 <= nbanks <= ANVIL_MAX_BANKS)
 *   d_scalars  DEVICE array of nbanks anvil_scalars read by the momentum kernel
 *              when it runs (so a captured CUDA graph sees the current values),
 *              or NULL to use banks[i].scalars, fixed at launch/capture time
 *   maps       host array of nmaps maps (1 <= nmaps <= ANVIL_MAX_MAPS), applied in order
 *   margin, eps  the normaliser d = sqrt(tr) * margin + eps (page: 1.05, 1e-6)
 *   workspace  DEVICE scratch of at least anvil_workspace_bytes(banks, nbanks)
 *              bytes, 256-byte aligned, owned by the caller; its contents on
 *              entry do not matter, and two calls that overlap on the GPU must
 *              not share it
 * Allocates nothing and never synchronises, so it may be captured in a CUDA graph. */
anvil_status anvil_multi_bank_step(const anvil_bank_desc* banks, int nbanks,
                                   const anvil_scalars* d_scalars,
                                   const anvil_map* maps, int nmaps, float margin, float eps,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* One bank with host scalars: the page's anvil_cascade signature with the slow
 * beta, the maps, margin and eps made parameters.  Uses a workspace owned by the
 * library, cached per device and grown on demand: a call that needs more than
 * the cached size frees and allocates it (cudaFree / cudaMalloc, which
 * synchronise the device), so make one call of the largest size before
 * capturing this function in a CUDA graph; a call that would have to grow it
 * while the stream is capturing returns ANVIL_ERR_WORKSPACE.  Every call on a
 * device uses that one workspace: two calls whose work can overlap on the GPU
 * (different streams, or threads) corrupt each other's results, so serialise
 * them, or give each stream its own workspace through anvil_multi_bank_step.
 * maps = NULL selects the page's six ANVIL_MAPS. */
anvil_status anvil_bank_step(const float* grad, float* velocity, int g, int m, int n,
                             float momentum, float fast_beta, float fast_weight, float slow_beta,
                             const anvil_map* maps, int nmaps, float margin, float eps,
                             uint16_t* out, void* stream);

/* anvil_bank_step for callers that must not allocate device memory.  The page has no
 * counterpart: this is a deployment convenience.  Some hosts cannot call cudaMalloc
 * from the code that runs the optimizer step: an application whose device memory is
 * all handed out by its own pool or budget, or a latency-bound loop where cudaMalloc /
 * cudaFree, which synchronise the device, are not allowed.  This variant takes the same arguments as
 * anvil_bank_step but keeps its scratch in a fixed array of
 * ANVIL_STATIC_SCRATCH_BYTES bytes of device memory that the library declares
 * statically: each GPU that loads the library holds that array until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Sizes whose scratch (anvil_workspace_bytes of the one bank) exceeds
 *     ANVIL_STATIC_SCRATCH_BYTES are rejected with ANVIL_ERR_WORKSPACE, and
 *     anvil_last_cuda_error() says how many bytes the call needed.  32 MiB holds,
 *     e.g., 22 matrices of 256 x 768 or 3 of 2816 x 768.
 *   - The first call on each GPU looks up the array's device address on that GPU
 *     (cudaGetSymbolAddress, with that GPU current); make that first call before
 *     any stream capture.
 *   - All calls on a GPU share the one array, which keeps whatever the last call
 *     left in it; the step writes every scratch byte before reading it, so nothing
 *     needs clearing.  Two calls whose work overlaps on the GPU (different streams,
 *     or threads) race on the array and corrupt each other's results: serialise them. */
#define ANVIL_STATIC_SCRATCH_BYTES (32u << 20)
anvil_status anvil_bank_step_noalloc(const float* grad, float* velocity, int g, int m, int n,
                                     float momentum, float fast_beta, float fast_weight,
                                     float slow_beta, const anvil_map* maps, int nmaps,
                                     float margin, float eps, uint16_t* out, void* stream);

/* ---- the update tail: anvil_bank_update's steps after the cascade on the page
 * (`_rail_equalizer`, then `_sign_aligned_decay_update`).  For every matrix, with the
 * bank step's output as the update v and lanes along the longer dimension (the rows
 * when m >= n, else the columns), each lane reduced over the other dimension:
 *   P[l] = mean over lane l of v^2;  lane_energy <- lerp(lane_energy, P, 1 - beta2)
 *   gain = rsqrt(max(lane_energy, 1e-10));  scale[l] = gain[l] * (||v||_F / post_norm),
 *   post_norm^2 = sum_l P[l] * lane_len * gain[l]^2   (post_norm clamped at 1e-10)
 *   u = bf16(v * bf16(scale[lane]))
 *   w = fp32 master weight (param bits << 16 | mantissa)
 *   w <- (w - w * [slow rail * w >= 0] * eff_wd * eff_lr[mat]) - u * eff_lr[mat]
 *   param, mantissa <- high and low 16 bits of w.
 * DEVICE pointers, row-major, caller-owned:
 *   update      [g, m, n] bf16 bits, read (the out of anvil_bank_step)
 *   velocity    [2, g, m, n] fp32, read (rail 1, the slow rail, gates the decay)
 *   lane_energy [g, m] fp32 if m >= n, else [g, n]; read and written
 *   param       [g, m, n] bf16 bits of the parameter; read and written
 *   mantissa    [g, m, n] uint16, the low half of the fp32 master weight; read and written
 *   eff_lr      [g] fp32 per-matrix learning rate, read when the kernels run
 *   tail_link   NULL, or the link buffer the step that produced `update` (its out) and
 *               `velocity` was given: the tail then takes the slow rail's signs from it,
 *               with the same results
 * Written buffers must not overlap any other buffer of the call. */
typedef struct {
    const uint16_t* update;
    const float* velocity;
    float* lane_energy;
    uint16_t* param;
    uint16_t* mantissa;
    const float* eff_lr;
    int g, m, n;
    float eff_wd, beta2;
    const void* tail_link;
} anvil_tail_desc;

/* Bytes of device workspace anvil_update_tail needs (0 if the descriptors are invalid). */
size_t anvil_tail_workspace_bytes(const anvil_tail_desc* banks, int nbanks);

/* The update tail over nbanks banks (1 <= nbanks <= ANVIL_MAX_BANKS), three grouped
 * launches on the stream;
 * workspace as for anvil_multi_bank_step (256-byte aligned, caller-owned, contents on
 * entry irrelevant).  Allocates nothing, never synchronises. */
anvil_status anvil_update_tail(const anvil_tail_desc* banks, int nbanks, void* workspace,
                               size_t workspace_bytes, void* stream);

/* The page's Adam step for the parameters outside the ANVIL banks (`_adam_update_step`:
 * bias-corrected Adam with cautious weight decay), elementwise over count fp32 values,
 * DEVICE pointers, caller-owned, read and written in place except grad:
 *   exp_avg    = exp_avg * beta1 + (1 - beta1) * grad
 *   exp_avg_sq = exp_avg_sq * beta2 + ((1 - beta2) * grad) * grad
 *   u = (exp_avg / (sqrt(exp_avg_sq) + eps)) * step_size
 *   u = u + (eff_wd * param) * [u * param > 0];   param = param - u
 * step_size (lr * sqrt(1 - beta2^t) / (1 - beta1^t)) and eff_wd are the caller's, as on
 * the page.  Buffers 4-byte aligned; param, exp_avg and exp_avg_sq must not overlap any
 * other buffer of the call.  One launch on the stream; allocates nothing. */
anvil_status anvil_adam_step(float* param, const float* grad, float* exp_avg, float* exp_avg_sq,
                             size_t count, float beta1, float beta2, float eps, float step_size,
                             float eff_wd, void* stream);

/* Per-stage dumps of one bank step, for parity testing (not the hot path).
 * DEVICE pointers, each optional (NULL = skip), in the page's layout:
 *   X_raw [g, m, n] bf16            bf16 cast of the momentum lookahead
 *   d     [g]       fp32            normaliser per matrix
 *   X     [nmaps+1, g, m, n] bf16   normalised X, then X after each map
 *   A, B  [nmaps, g, s, s] bf16     per map (s = min(m, n)); A[0] is the
 *                                   normalised first Gram */
typedef struct {
    uint16_t* X_raw;
    float* d;
    uint16_t* X;
    uint16_t* A;
    uint16_t* B;
} anvil_trace;

/* anvil_multi_bank_step for one bank, plus the dumps.  Same arguments and
 * workspace rules; out receives the same result as without tracing.  The cascade
 * runs one phase per launch here (with the dumps copied out in between); a trace
 * with every pointer NULL gives that phase-by-phase run without dumps. */
anvil_status anvil_bank_step_traced(const anvil_bank_desc* bank, const anvil_scalars* d_scalars,
                                    const anvil_map* maps, int nmaps, float margin, float eps,
                                    void* workspace, size_t workspace_bytes,
                                    const anvil_trace* trace, void* stream);

/* Reads (and, if clear != 0, resets) the current device's error word, which a
 * kernel sets when one of its bounded waits gives up instead of hanging.
 * Synchronises the device.  Returns ANVIL_OK, ANVIL_ERR_TIMEOUT or ANVIL_ERR_CUDA. */
anvil_status anvil_device_error(int clear);

/* The error word as the work queued so far on `stream` leaves it: waits for that stream
 * only (cudaStreamSynchronize), then reads and resets the word with one atomic exchange
 * on the device, so a timeout is reported once.  The word belongs to the device, not to
 * the stream: a wait that gave up in work on another stream shows here too if it gave up
 * before this read, and otherwise in a later read.  Returns ANVIL_OK, ANVIL_ERR_TIMEOUT,
 * ANVIL_ERR_CUDA or ANVIL_ERR_DEVICE. */
anvil_status anvil_last_device_error(void* stream);

/* Self-test of the bounded waits: launches one block that waits on a barrier
 * nothing will ever complete, for at most timeout_us microseconds, after which
 * it records a timeout in the device error word and returns.  It neither
 * faults nor hangs the GPU. */
anvil_status anvil_selftest_wait_timeout(unsigned timeout_us, void* stream);

/* Per-launch timing for benchmarks.  Between anvil_profile_begin and
 * anvil_profile_end, every kernel launch of anvil_multi_bank_step, anvil_bank_step,
 * anvil_update_tail and anvil_adam_step in the process is bracketed by two CUDA events
 * recorded on the call's stream (at most max_records launches; later ones are
 * not timed).  begin creates the events (a host call: do not begin, or step
 * with profiling on, while a stream is capturing).  end synchronises, writes up
 * to cap records in launch order, destroys the events and returns how many
 * launches were timed (negative on a CUDA error). */
/* Kinds 3-7 are the cascade's phases, each its own launch in traced steps only; an
 * untraced step runs them all in one ANVIL_KERNEL_CASCADE launch. */
typedef enum {
    ANVIL_KERNEL_MOMENTUM = 0,     /* momentum + cast + diagonal partials */
    ANVIL_KERNEL_NORM_D = 1,       /* d per matrix */
    ANVIL_KERNEL_NORMALIZE = 2,    /* X <- bf16(X / d) */
    ANVIL_KERNEL_GRAM_NORM = 3,    /* first Gram, A = bf16(bf16(X X^T) / d^2) */
    ANVIL_KERNEL_GRAM = 4,         /* A = bf16(X X^T) */
    ANVIL_KERNEL_SQPOLY = 5,       /* B = bf16(b A + c A A) */
    ANVIL_KERNEL_XUPDATE = 6,      /* X <- bf16(a X + B X) */
    ANVIL_KERNEL_XUPDATE_OUT = 7,  /* the last map's X-update, written to out */
    ANVIL_KERNEL_TAIL_POWER = 8,   /* update tail: lane powers */
    ANVIL_KERNEL_TAIL_SCALE = 9,   /* update tail: lane energies and scales */
    ANVIL_KERNEL_TAIL_APPLY = 10,  /* update tail: equalise + sign-aligned decay update */
    ANVIL_KERNEL_ADAM = 11,        /* Adam step */
    ANVIL_KERNEL_CASCADE = 12      /* the whole cascade (every product of every map) */
} anvil_kernel_kind;

typedef struct { int kind; float ms; } anvil_profile_record;

anvil_status anvil_profile_begin(int max_records);
int anvil_profile_end(anvil_profile_record* records, int cap);

/* Diagnostic, host only (no CUDA call, no GPU needed): the order in which the cascade
 * kernel of anvil_multi_bank_step walks its work items for these banks and nmaps maps.
 * Items are 256 x 256 output tiles; the kernel's phases are the first Gram, then per
 * map the Gram (after the first map), B = bA + cA^2 and the X-update (the normalisation
 * X / d is its own kernel, before the cascade).  The order is a list of runs, each one phase of a range of matrices of one
 * bank, matrix by matrix; every phase of a matrix comes after the phases it reads.
 * Writes up to cap runs and returns how many there are (-1 on invalid arguments). */
typedef struct {
    int phase;  /* phase index, 0 = the first Gram */
    int op;     /* 0 Gram, 1 first Gram, 2 B = bA + cA^2, 3 X-update, 4 last X-update */
    int bank;   /* index of the bank in the call */
    int mat0;   /* first matrix of the run */
    int nmat;   /* matrices in the run */
    int begin;  /* index of the run's first item in the walk */
    int tiles;  /* items per matrix in this phase */
} anvil_schedule_run;
int anvil_schedule_runs(const anvil_bank_desc* banks, int nbanks, int nmaps, anvil_schedule_run* runs, int cap);

/* Per-item timeline of the cascade kernel, for performance work.  Only a library built
 * with the timeline option (build.py --timeline, which writes libanvil_timeline.so)
 * records it; this library returns ANVIL_ERR_UNAVAILABLE.  Item t (0-based, in the
 * order of anvil_schedule_runs) of the latest cascade launch owns 16 64-bit words
 * starting at word 16 t, for t < ANVIL_TIMELINE_ITEMS:
 *   0 pair | (op | bank << 8 | phase << 16) << 16 | matrix << 48;  1 block row | block
 *   column << 16 | k-blocks << 32;  then %globaltimer nanoseconds when 2 the pair's
 *   scheduler took it, 3 its input phases were complete, 4 its entry was handed out,
 *   5 the first operand load was armed, 6 the MMA issuer read it, 7 its accumulator was
 *   free, 8 its first k-block landed, 9 its last MMAs were issued, 10 the epilogue found
 *   the accumulator complete, 11 the epilogue was done;  12 and 13: SM cycles (clock64)
 *   at 8 and 9;  14 SM cycles the MMA issuer waited for k-blocks after the first to
 *   land;  15 SM cycles the producer waited for free operand stages.
 * anvil_timeline_read copies min(bytes, the buffer) to host memory (synchronous; call
 * after the launch has completed).  anvil_timeline_clear zeroes the buffer. */
#define ANVIL_TIMELINE_ITEMS 16384
anvil_status anvil_timeline_read(void* host, size_t bytes);
anvil_status anvil_timeline_clear(void);

/* Human-readable name of a status. */
const char* anvil_status_string(anvil_status status);

/* Text of the last CUDA error this library saw on this thread ("" if none). */
const char* anvil_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ANVIL_H */
