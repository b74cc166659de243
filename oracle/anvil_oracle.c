/*
 * anvil_oracle.c -- the CPU oracle of the ANVIL bank step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the bench's cpu_baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes follows the page "modded-nanogpt track_1_short/optim/anvil.py",
 * function `anvil_cascade` (twin-rail Nesterov momentum, then the whitening
 * cascade driven by ANVIL_MAPS), step by step and in the page's order:
 *
 *   g  = float(grad_chunk)
 *   velocity[0] <- lerp(velocity[0], g, 1 - fast_beta)      (fast rail)
 *   velocity[1] <- lerp(velocity[1], g, 1 - slow_beta)      (slow rail)
 *   blend = w * velocity[0] + (1 - w) * velocity[1]
 *   g  <- lerp(g, blend, momentum)
 *   X  = bf16(g);  is_tall = rows > cols
 *   A  = bf16(Gram(X))    tall: X^T X,  wide (square included): X X^T
 *   tr = sum_i float(A[i,i]);  d = sqrt(tr) * margin + eps
 *   X  = bf16(float(X) / d);  A = bf16(float(A) / d^2)
 *   for k, (a, b, c) in maps:
 *       if k > 0: A = bf16(Gram(X))
 *       B = bf16(b * A + c * (A @ A))
 *       X = bf16(a * X + X @ B)    (tall)      X = bf16(a * X + B @ X)    (wide)
 *
 * Precision reading: every tensor the page stores as bf16 (X, A, B, C) is
 * rounded to bf16 round-to-nearest-even; everything in between is fp32 with one
 * rounding per operation (compiled with -ffp-contract=off); matrix products sum
 * their fp32 products sequentially in k order (the products of two bf16 values
 * are exact in fp32).  lerp(s, e, w) = s + w * (e - s).  The page's split
 * baddbmm form (two roundings for banks over 1024 rows) is available behind the
 * `split` flag only to measure its effect; the default is one rounding.
 *
 * A parallel fp64 iteration (`oracle_cascade_f64`) runs the same steps with no
 * rounding at all, for the SVD closed-form pin.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define EXPORT __attribute__((visibility("default")))

/* ---- bf16 storage, written from the IEEE-754 binary32 / bfloat16 layouts ----
 * bfloat16 is the top 16 bits of a binary32.  Rounding to nearest, ties to
 * even, on the 16 dropped bits: add 0x7FFF plus the lowest kept bit, then
 * truncate.  A carry out of the mantissa correctly bumps the exponent (and
 * turns the largest finite values into infinity).  NaNs keep their sign and
 * top payload bits and are forced quiet. */
static inline float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static inline float round_bf16(float f) { return bf16_to_f32(f32_to_bf16(f)); }

EXPORT void oracle_f32_to_bf16(const float* in, uint16_t* out, long count) {
    for (long i = 0; i < count; ++i) out[i] = f32_to_bf16(in[i]);
}

/* ---- plain fp32 matrix product with sequential k-order sums ----
 * C[i][j] = sum_{k=0..K-1} A[i][k] * B[k][j], all row-major, fp32 accumulate.
 * Each output is summed in increasing k (the loop order i,k,j keeps that); rows
 * are independent, so OpenMP over i does not change any sum. */
static void matmul_f32(const float* A, const float* B, float* C, int M, int K, int N) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        float* c = C + (size_t)i * N;
        for (int j = 0; j < N; ++j) c[j] = 0.0f;
        const float* a = A + (size_t)i * K;
        for (int k = 0; k < K; ++k) {
            const float aik = a[k];
            const float* b = B + (size_t)k * N;
            for (int j = 0; j < N; ++j) c[j] += aik * b[j];
        }
    }
}

static void transpose_f32(const float* A, float* T, int rows, int cols) {
    for (int i = 0; i < rows; ++i)
        for (int j = 0; j < cols; ++j) T[(size_t)j * rows + i] = A[(size_t)i * cols + j];
}

static void to_f32(const uint16_t* h, float* f, size_t n) {
    for (size_t i = 0; i < n; ++i) f[i] = bf16_to_f32(h[i]);
}

static void to_bf16(const float* f, uint16_t* h, size_t n) {
    for (size_t i = 0; i < n; ++i) h[i] = f32_to_bf16(f[i]);
}

/* ---- twin-rail Nesterov momentum (anvil_cascade, first block) ----
 * grad: count fp32 values (read only; the page lerps a float copy of it).
 * v_fast, v_slow: the two rails, updated in place.
 * g_out (optional): the fp32 lookahead; X_out (optional): bf16(g). */
static inline float lerp32(float s, float e, float w) { return s + w * (e - s); }

EXPORT void oracle_momentum(const float* grad, float* v_fast, float* v_slow, long count,
                            float momentum, float fast_beta, float fast_weight, float slow_beta,
                            float* g_out, uint16_t* X_out) {
    const float w_fast = 1.0f - fast_beta;
    const float w_slow = 1.0f - slow_beta;
    const float w = fast_weight;
    const float one_minus_w = 1.0f - w;
#pragma omp parallel for schedule(static)
    for (long e = 0; e < count; ++e) {
        float g = grad[e];
        float v0 = lerp32(v_fast[e], g, w_fast);
        float v1 = lerp32(v_slow[e], g, w_slow);
        v_fast[e] = v0;
        v_slow[e] = v1;
        float blend = w * v0 + one_minus_w * v1;
        g = lerp32(g, blend, momentum);
        if (g_out) g_out[e] = g;
        if (X_out) X_out[e] = f32_to_bf16(g);
    }
}

/* ---- one Gram, bf16 in and out ----
 * tall (rows > cols): A = X^T X, s = cols;  wide: A = X X^T, s = rows. */
static void gram_bf16(const float* Xf, int rows, int cols, int is_tall, float* scratchT,
                      float* Af32, uint16_t* A) {
    const int s = is_tall ? cols : rows;
    if (is_tall) {
        transpose_f32(Xf, scratchT, rows, cols);             /* X^T: [cols, rows] */
        matmul_f32(scratchT, Xf, Af32, cols, rows, cols);    /* X^T @ X */
    } else {
        transpose_f32(Xf, scratchT, rows, cols);             /* X^T: [cols, rows] */
        matmul_f32(Xf, scratchT, Af32, rows, cols, rows);    /* X @ X^T */
    }
    to_bf16(Af32, A, (size_t)s * s);
}

/* Optional per-stage dumps, all bf16 bits in the page's layout:
 *   trace_A0 [s*s]        the first Gram before normalisation
 *   trace_X  [(nmaps+1) * rows*cols]  X after normalisation, then after each map
 *   trace_A  [nmaps * s*s], trace_B [nmaps * s*s]  per map
 *   trace_d  [1]  (fp32) */
typedef struct {
    uint16_t* A0;
    uint16_t* X;
    uint16_t* A;
    uint16_t* B;
    float* d;
} oracle_trace;

/* The cascade on one matrix.  X_in, X_out: bf16 bits [rows, cols] (may alias).
 * maps: nmaps triples (a, b, c) as fp32.  Returns 0, or -1 on allocation failure. */
EXPORT int oracle_cascade(const uint16_t* X_in, int rows, int cols, const float* maps, int nmaps,
                          float margin, float eps, int split, uint16_t* X_out,
                          const oracle_trace* trace) {
    const int is_tall = rows > cols;
    const int s = is_tall ? cols : rows;
    const size_t nX = (size_t)rows * cols, nA = (size_t)s * s;
    float* Xf = malloc(nX * sizeof(float));
    float* Cf = malloc(nX * sizeof(float));
    float* T = malloc(nX * sizeof(float));
    float* Af = malloc(nA * sizeof(float));
    float* Bf = malloc(nA * sizeof(float));
    float* P = malloc(nA * sizeof(float));
    uint16_t* A = malloc(nA * sizeof(uint16_t));
    uint16_t* B = malloc(nA * sizeof(uint16_t));
    uint16_t* X = malloc(nX * sizeof(uint16_t));
    if (!Xf || !Cf || !T || !Af || !Bf || !P || !A || !B || !X) {
        free(Xf); free(Cf); free(T); free(Af); free(Bf); free(P); free(A); free(B); free(X);
        return -1;
    }
    memcpy(X, X_in, nX * sizeof(uint16_t));
    to_f32(X, Xf, nX);

    /* The first Gram is taken on the unnormalised X; its bf16 diagonal gives the trace. */
    gram_bf16(Xf, rows, cols, is_tall, T, Af, A);
    if (trace && trace->A0) memcpy(trace->A0, A, nA * sizeof(uint16_t));
    float tr = 0.0f;
    for (int i = 0; i < s; ++i) tr += bf16_to_f32(A[(size_t)i * s + i]);
    const float d = sqrtf(tr) * margin + eps;
    const float d2 = d * d;
    if (trace && trace->d) trace->d[0] = d;
    for (size_t e = 0; e < nX; ++e) X[e] = f32_to_bf16(bf16_to_f32(X[e]) / d);
    for (size_t e = 0; e < nA; ++e) A[e] = f32_to_bf16(bf16_to_f32(A[e]) / d2);
    to_f32(X, Xf, nX);
    if (trace && trace->X) memcpy(trace->X, X, nX * sizeof(uint16_t));

    for (int k = 0; k < nmaps; ++k) {
        const float a = maps[3 * k], b = maps[3 * k + 1], c = maps[3 * k + 2];
        if (k > 0) gram_bf16(Xf, rows, cols, is_tall, T, Af, A);
        /* B = b * A + c * (A @ A) */
        to_f32(A, Af, nA);
        matmul_f32(Af, Af, P, s, s, s);
        for (size_t e = 0; e < nA; ++e) Bf[e] = b * Af[e] + c * P[e];
        to_bf16(Bf, B, nA);
        to_f32(B, Bf, nA);
        /* C = a * X + X @ B (tall) or a * X + B @ X (wide) */
        if (is_tall) matmul_f32(Xf, Bf, Cf, rows, cols, cols);
        else matmul_f32(Bf, Xf, Cf, rows, rows, cols);
        if (split) {
            for (size_t e = 0; e < nX; ++e) Cf[e] = round_bf16(Cf[e]);
            for (size_t e = 0; e < nX; ++e) X[e] = f32_to_bf16(Cf[e] + a * Xf[e]);
        } else {
            for (size_t e = 0; e < nX; ++e) X[e] = f32_to_bf16(a * Xf[e] + Cf[e]);
        }
        to_f32(X, Xf, nX);
        if (trace && trace->A) memcpy(trace->A + (size_t)k * nA, A, nA * sizeof(uint16_t));
        if (trace && trace->B) memcpy(trace->B + (size_t)k * nA, B, nA * sizeof(uint16_t));
        if (trace && trace->X) memcpy(trace->X + (size_t)(k + 1) * nX, X, nX * sizeof(uint16_t));
    }
    memcpy(X_out, X, nX * sizeof(uint16_t));
    free(Xf); free(Cf); free(T); free(Af); free(Bf); free(P); free(A); free(B); free(X);
    return 0;
}

/* ---- the same iteration in fp64 with no rounding at all (for the SVD closed form) ---- */
static void matmul_f64(const double* A, const double* B, double* C, int M, int K, int N) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; ++i) {
        double* c = C + (size_t)i * N;
        for (int j = 0; j < N; ++j) c[j] = 0.0;
        const double* a = A + (size_t)i * K;
        for (int k = 0; k < K; ++k) {
            const double aik = a[k];
            const double* b = B + (size_t)k * N;
            for (int j = 0; j < N; ++j) c[j] += aik * b[j];
        }
    }
}

EXPORT int oracle_cascade_f64(const double* X_in, int rows, int cols, const double* maps,
                              int nmaps, double margin, double eps, double* X_out) {
    const int is_tall = rows > cols;
    const int s = is_tall ? cols : rows;
    const size_t nX = (size_t)rows * cols, nA = (size_t)s * s;
    double* X = malloc(nX * sizeof(double));
    double* C = malloc(nX * sizeof(double));
    double* T = malloc(nX * sizeof(double));
    double* A = malloc(nA * sizeof(double));
    double* B = malloc(nA * sizeof(double));
    double* P = malloc(nA * sizeof(double));
    if (!X || !C || !T || !A || !B || !P) {
        free(X); free(C); free(T); free(A); free(B); free(P);
        return -1;
    }
    memcpy(X, X_in, nX * sizeof(double));
    for (int i = 0; i < rows; ++i)
        for (int j = 0; j < cols; ++j) T[(size_t)j * rows + i] = X[(size_t)i * cols + j];
    if (is_tall) matmul_f64(T, X, A, cols, rows, cols);
    else matmul_f64(X, T, A, rows, cols, rows);
    double tr = 0.0;
    for (int i = 0; i < s; ++i) tr += A[(size_t)i * s + i];
    const double d = sqrt(tr) * margin + eps;
    for (size_t e = 0; e < nX; ++e) X[e] /= d;
    for (size_t e = 0; e < nA; ++e) A[e] /= d * d;
    for (int k = 0; k < nmaps; ++k) {
        const double a = maps[3 * k], b = maps[3 * k + 1], c = maps[3 * k + 2];
        if (k > 0) {
            for (int i = 0; i < rows; ++i)
                for (int j = 0; j < cols; ++j) T[(size_t)j * rows + i] = X[(size_t)i * cols + j];
            if (is_tall) matmul_f64(T, X, A, cols, rows, cols);
            else matmul_f64(X, T, A, rows, cols, rows);
        }
        matmul_f64(A, A, P, s, s, s);
        for (size_t e = 0; e < nA; ++e) B[e] = b * A[e] + c * P[e];
        if (is_tall) matmul_f64(X, B, C, rows, cols, cols);
        else matmul_f64(B, X, C, rows, rows, cols);
        for (size_t e = 0; e < nX; ++e) X[e] = a * X[e] + C[e];
    }
    memcpy(X_out, X, nX * sizeof(double));
    free(X); free(C); free(T); free(A); free(B); free(P);
    return 0;
}

/* ---- one bank: g matrices [g, rows, cols], velocity [2, g, rows, cols] ----
 * grad fp32 (read only), velocity fp32 in/out, out bf16 bits [g, rows, cols]. */
EXPORT int oracle_bank_step(const float* grad, float* velocity, int g, int rows, int cols,
                            float momentum, float fast_beta, float fast_weight, float slow_beta,
                            const float* maps, int nmaps, float margin, float eps, int split,
                            uint16_t* out) {
    const size_t nX = (size_t)rows * cols, count = (size_t)g * nX;
    uint16_t* X = malloc(count * sizeof(uint16_t));
    if (!X) return -1;
    oracle_momentum(grad, velocity, velocity + count, (long)count, momentum, fast_beta,
                    fast_weight, slow_beta, NULL, X);
    int rc = 0;
    for (int i = 0; i < g && rc == 0; ++i)
        rc = oracle_cascade(X + i * nX, rows, cols, maps, nmaps, margin, eps, split,
                            out + i * nX, NULL);
    free(X);
    return rc;
}

/* ---- the update tail: anvil.py, `_rail_equalizer` and `_sign_aligned_decay_update` ----
 *
 * Equaliser, per matrix of a bank [g, rows, cols] of bf16 updates v (the cascade output):
 * lanes run along the longer dimension (rows when rows >= cols, else columns) and each
 * lane is reduced over the other one, of length lane_len:
 *   lane_power[l] = mean over the lane of float(v)^2
 *   pre_norm      = sqrt(sum_l lane_power[l] * lane_len)          (= ||v||_F)
 *   lane_energy   <- lerp(lane_energy, lane_power, 1 - beta2)      (fp32 state)
 *   gain[l]       = rsqrt(max(lane_energy[l], 1e-10))
 *   post_power[l] = (lane_power[l] * lane_len) * gain[l]^2
 *   post_norm     = sqrt(sum_l post_power[l])
 *   scale[l]      = gain[l] * (pre_norm / max(post_norm, 1e-10))
 *   v_eq          = bf16(float(v) * float(bf16(scale[lane])))      (scale cast to v's dtype)
 * Sums run sequentially in fp32; mean = sum / lane_len; rsqrt is the correctly rounded
 * 1/sqrt; one rounding per operation as elsewhere. */
static inline float rsqrt_rn(float x) { return (float)(1.0 / sqrt((double)x)); }

EXPORT void oracle_rail_equalizer(const uint16_t* v, int g, int rows, int cols, float* lane_energy,
                                  float beta2, uint16_t* v_eq) {
    const int lanes_are_rows = rows >= cols;
    const int nl = lanes_are_rows ? rows : cols;
    const int lane_len = lanes_are_rows ? cols : rows;
    const float w = 1.0f - beta2;
    float* power = malloc((size_t)nl * sizeof(float));
    float* scale = malloc((size_t)nl * sizeof(float));
    for (int mtx = 0; mtx < g; ++mtx) {
        const uint16_t* V = v + (size_t)mtx * rows * cols;
        uint16_t* E = v_eq + (size_t)mtx * rows * cols;
        float* le = lane_energy + (size_t)mtx * nl;
        for (int l = 0; l < nl; ++l) {
            float s = 0.0f;
            for (int k = 0; k < lane_len; ++k) {
                const float x = bf16_to_f32(lanes_are_rows ? V[(size_t)l * cols + k] : V[(size_t)k * cols + l]);
                s += x * x;
            }
            power[l] = s / (float)lane_len;
        }
        float psum = 0.0f;
        for (int l = 0; l < nl; ++l) psum += power[l];
        const float pre_norm = sqrtf(psum * (float)lane_len);
        float qsum = 0.0f;
        for (int l = 0; l < nl; ++l) {
            le[l] = lerp32(le[l], power[l], w);
            const float gain = rsqrt_rn(le[l] > 1e-10f ? le[l] : 1e-10f);
            const float post = (power[l] * (float)lane_len) * (gain * gain);
            qsum += post;
            scale[l] = gain;
        }
        float post_norm = sqrtf(qsum);
        if (post_norm < 1e-10f) post_norm = 1e-10f;
        const float ratio = pre_norm / post_norm;
        for (int l = 0; l < nl; ++l) scale[l] = round_bf16(scale[l] * ratio);
        for (int i = 0; i < rows; ++i)
            for (int j = 0; j < cols; ++j) {
                const size_t e = (size_t)i * cols + j;
                E[e] = f32_to_bf16(bf16_to_f32(V[e]) * scale[lanes_are_rows ? i : j]);
            }
    }
    free(power);
    free(scale);
}

/* Sign-aligned decay + parameter update on the fp32 master weight held as bf16 bits p
 * (high half) and mantissa (low half), elementwise over g matrices of `count` elements:
 *   w       = float(p << 16 | mantissa)
 *   aligned = float(gate) * w >= 0          (gate: the slow rail)
 *   w       = (w - ((w * aligned) * wd) * lr[mtx]) - update * lr[mtx]
 *   p, mantissa = high and low 16 bits of w (a bit split, no rounding) */
EXPORT void oracle_sign_aligned_decay(uint16_t* p, uint16_t* mantissa, const uint16_t* update,
                                      const float* gate, int g, long count, float wd,
                                      const float* lr) {
    for (int mtx = 0; mtx < g; ++mtx) {
        const float lrm = lr[mtx];
        for (long k = 0; k < count; ++k) {
            const size_t e = (size_t)mtx * count + k;
            uint32_t bits = ((uint32_t)p[e] << 16) | mantissa[e];
            float w;
            memcpy(&w, &bits, 4);
            const float aligned = (gate[e] * w >= 0.0f) ? 1.0f : 0.0f;
            const float u = bf16_to_f32(update[e]);
            w = (w - ((w * aligned) * wd) * lrm) - u * lrm;
            memcpy(&bits, &w, 4);
            p[e] = (uint16_t)(bits >> 16);
            mantissa[e] = (uint16_t)(bits & 0xFFFFu);
        }
    }
}

/* ---- Adam with cautious weight decay: anvil.py, `_adam_update_step` ----
 * Elementwise over count fp32 values, the page's tensor operations in order, one rounding
 * each (step_size = lr * sqrt(1 - beta2^t) / (1 - beta1^t) and eff_wd are the caller's):
 *   exp_avg    = exp_avg * beta1 + (1 - beta1) * g
 *   exp_avg_sq = exp_avg_sq * beta2 + ((1 - beta2) * g) * g
 *   update     = (exp_avg / (sqrt(exp_avg_sq) + eps)) * step_size
 *   update     = update + (eff_wd * p) * [update * p > 0]
 *   p          = p - update */
EXPORT void oracle_adam_step(float* p, const float* g, float* exp_avg, float* exp_avg_sq, long count,
                             float beta1, float beta2, float eps, float step_size, float eff_wd) {
    const float c1 = 1.0f - beta1, c2 = 1.0f - beta2;
    for (long e = 0; e < count; ++e) {
        const float m = exp_avg[e] * beta1 + c1 * g[e];
        const float v = exp_avg_sq[e] * beta2 + (c2 * g[e]) * g[e];
        exp_avg[e] = m;
        exp_avg_sq[e] = v;
        float u = (m / (sqrtf(v) + eps)) * step_size;
        const float mask = (u * p[e] > 0.0f) ? 1.0f : 0.0f;
        u = u + (eff_wd * p[e]) * mask;
        p[e] = p[e] - u;
    }
}

EXPORT int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

EXPORT void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
