/*
 * FP64 CPU oracle for the fused linear log-probability operator and the
 * deterministic GEMM family (fwd, dA, dB).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg may load this library.  The
 * product path (the CUDA library and its Python binding) never calls it and
 * shares no code, header, table or constant with it.
 *
 * Every result is the plain mathematical definition evaluated in double
 * precision over the BF16-rounded inputs; there is no tiling, no vocabulary
 * split, no online softmax and no reordering beyond what each definition
 * states.  Rows are independent, so OpenMP spreads rows over threads; each
 * row's arithmetic is the same sequence whatever the thread count.
 *
 * Sources (web pages of the RL-Kernel project):
 *   [P3] "feat(linear-logp): add batch-invariant fused SM90 operator" —
 *        Walkthrough (hidden . W^T -> log-sum-exp -> target gather, returning
 *        log-probability and log-sum-exp) and the PR body (the split + online
 *        softmax + combine path is equivalent in real arithmetic to this
 *        definition).
 *   [P1] "feat(musa): add native deterministic gemm kernel" — Summary
 *        (forward C = A B, dA = dC B^T, dB = A^T dC, FP32 accumulation in a
 *        fixed ascending K order) and the review comment on the FP32-output
 *        backward (grad_output is cast to BF16 before dA / dB).
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * No contraction into FMA and no fast-math, so every double operation rounds
 * exactly as written.
 *
 * Parity pins (what checks this file against something other than itself)
 * live in tests/test_oracle_pins.py: 50-digit brute force, torch float64
 * library routines, closed forms and invariants, exact integer GEMMs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ORACLE_MUTANT selects a deliberately planted mistake so that the pin suite
 * can show that it catches it.  0 (the default) is the correct oracle.
 *   1: bias dropped from the logits     2: last hidden term of each logit dropped
 *   3: log-sum-exp loses its max term   4: logp sign flipped
 *   5: forward reads B transposed       6: dA reads B as if it were [N, K]
 *      (square operands only)              (square operands only)
 *   7: dB drops the last row of A / dC  8: BF16 rounding sends ties away from 0
 *   9: dL/dz sign flipped              10: dL/dz loses its one-hot term          */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---- BF16 / FP32 bit conversions (the oracle's own) -------------------- */

/* A BF16 value is the upper 16 bits of an IEEE binary32; decoding is exact. */
static double bf16_decode(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_bf16_to_f64(uint16_t b) { return bf16_decode(b); }

/* binary32 -> BF16, round to nearest, ties to even; NaN stays NaN (quiet). */
uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xffffu;
    uint32_t upper = u >> 16;
    uint32_t half = 0x8000u;
#if ORACLE_MUTANT == 8
    if (lower >= half) upper += 1u;
#else
    if (lower > half || (lower == half && (upper & 1u))) upper += 1u;
#endif
    return (uint16_t)upper;
}

void oracle_f32_to_bf16_rne_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16_rne(in[i]);
}

/* double -> BF16 with a single rounding (no detour through binary32, which
 * would round twice).  BF16 keeps 8 significant bits; its normal range starts
 * at 2^-126 and its subnormal quantum is 2^-133. */
uint16_t oracle_f64_to_bf16_rne(double x) {
    if (isnan(x)) return 0x7fc0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int qe = e - 8;
    if (qe < -133) qe = -133;
    double n = ldexp(a, -qe);           /* exact: scaling by a power of two */
    double r = nearbyint(n);            /* default mode: nearest, ties to even */
    double y = ldexp(r, qe);
    if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7f80u);
    float yf = (float)y;                /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &yf, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void oracle_f64_to_bf16_rne_array(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16_rne(in[i]);
}

static int set_threads(int n_threads) {
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
    return omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- linear log-probability [P3 Walkthrough] ---------------------------- */

/* z[v] = sum_h x[r,h] * w[v,h] (ascending h) + bias[v]. */
static void logits_row(const uint16_t* x, int64_t H, const uint16_t* weight, int64_t ld_w,
                       int64_t V, const float* bias, double* z) {
    for (int64_t v = 0; v < V; ++v) {
        const uint16_t* w = weight + v * ld_w;
        double acc = 0.0;
#if ORACLE_MUTANT == 2
        int64_t h_end = H - 1;
#else
        int64_t h_end = H;
#endif
        for (int64_t h = 0; h < h_end; ++h) acc += bf16_decode(x[h]) * bf16_decode(w[h]);
#if ORACLE_MUTANT != 1
        if (bias) acc += (double)bias[v];
#endif
        z[v] = acc;
    }
}

/* All N x V logits (small cases only). */
void oracle_logits(const uint16_t* hidden, int64_t N, int64_t H, int64_t ld_h,
                   const uint16_t* weight, int64_t V, int64_t ld_w, const float* bias,
                   double* z /* [N, V] */) {
    for (int64_t r = 0; r < N; ++r)
        logits_row(hidden + r * ld_h, H, weight, ld_w, V, bias, z + r * V);
}

/* lse = log(sum_v exp(z_v)), evaluated as M + log(sum_v exp(z_v - M)) with
 * M = max_v z_v so that no term overflows. */
static double logsumexp(const double* z, int64_t V) {
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if (z[v] > M) M = z[v];
    double s = 0.0;
#if ORACLE_MUTANT == 3
    for (int64_t v = 0; v < V; ++v) s += exp(z[v] - M);
    return log(s);
#else
    for (int64_t v = 0; v < V; ++v) s += exp(z[v] - M);
    return M + log(s);
#endif
}

/*
 * For each selected row r = rows[i] (all rows 0..N-1 when rows == NULL):
 *   lse[i]  = log sum_v exp(z_v)
 *   logp[i] = z_{target[r]} - lse[i]     (NaN when target[r] is not in [0, V))
 *   zt[i]   = z_{target[r]}              (NaN likewise; may be NULL)
 * target is read as target[r * target_stride] (stride 0 = one shared id).
 * Returns 0, or -1 when scratch memory cannot be allocated.
 */
int oracle_linear_logp(const uint16_t* hidden, int64_t N, int64_t H, int64_t ld_h,
                       const uint16_t* weight, int64_t V, int64_t ld_w, const float* bias,
                       const int64_t* target, int64_t target_stride,
                       const int64_t* rows, int64_t n_rows,
                       double* logp, double* lse, double* zt, int n_threads) {
    int64_t count = rows ? n_rows : N;
    int failed = 0;
    set_threads(n_threads);
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)(V > 0 ? V : 1) * sizeof(double));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t i = 0; i < count; ++i) {
            if (!z) continue;
            int64_t r = rows ? rows[i] : i;
            logits_row(hidden + r * ld_h, H, weight, ld_w, V, bias, z);
            double l = logsumexp(z, V);
            int64_t t = target[r * target_stride];
            double zv = (t >= 0 && t < V) ? z[t] : NAN;
#if ORACLE_MUTANT == 4
            logp[i] = l - zv;
#else
            logp[i] = zv - l;
#endif
            lse[i] = l;
            if (zt) zt[i] = zv;
        }
        free(z);
    }
    return failed ? -1 : 0;
}

/*
 * Gradient of the loss L = sum_r g[r] * logp[r] with respect to the logits:
 *   G[r, v] = dL/dz[r, v] = g[r] * ([v == t_r] - exp(z[r, v] - lse[r]))
 * (the derivative of log_softmax(z)[t] is onehot(t) - softmax(z)).  A row whose
 * target is outside [0, V) has no log-probability and gets a zero row.
 * Writes all N x V entries of G (small cases only).  Returns 0, or -1 when
 * scratch memory cannot be allocated.
 */
int oracle_linear_logp_grad_logits(const uint16_t* hidden, int64_t N, int64_t H, int64_t ld_h,
                                   const uint16_t* weight, int64_t V, int64_t ld_w,
                                   const float* bias, const int64_t* target,
                                   int64_t target_stride, const double* g, double* G,
                                   int n_threads) {
    int failed = 0;
    set_threads(n_threads);
#pragma omp parallel
    {
        double* z = (double*)malloc((size_t)(V > 0 ? V : 1) * sizeof(double));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < N; ++r) {
            if (!z) continue;
            double* Gr = G + r * V;
            int64_t t = target[r * target_stride];
            if (t < 0 || t >= V) {
                for (int64_t v = 0; v < V; ++v) Gr[v] = 0.0;
                continue;
            }
            logits_row(hidden + r * ld_h, H, weight, ld_w, V, bias, z);
            double l = logsumexp(z, V);
            for (int64_t v = 0; v < V; ++v) {
                double p = exp(z[v] - l);
#if ORACLE_MUTANT == 9
                Gr[v] = g[r] * (p - (v == t ? 1.0 : 0.0));
#elif ORACLE_MUTANT == 10
                Gr[v] = g[r] * (0.0 - p);
#else
                Gr[v] = g[r] * ((v == t ? 1.0 : 0.0) - p);
#endif
            }
        }
        free(z);
    }
    return failed ? -1 : 0;
}

/* ---- deterministic GEMM family [P1 Summary] ----------------------------- */
/* Every output element is one dot product over the reduction index taken in
 * ascending order, in double.  The loops walk a whole output row at a time
 * (i-k-j order) for cache locality; each element still sees its terms in
 * ascending reduction order. */

/* C[i, :] = sum_k A[i, k] * B[k, :] for the selected rows i of A [M, K], B [K, N]. */
void oracle_gemm_fwd(const uint16_t* A, int64_t M, int64_t K, int64_t lda,
                     const uint16_t* B, int64_t N, int64_t ldb,
                     const int64_t* rows, int64_t n_rows, double* C /* [count, N] */,
                     int n_threads) {
    int64_t count = rows ? n_rows : M;
    set_threads(n_threads);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        int64_t r = rows ? rows[i] : i;
        double* c = C + i * N;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = bf16_decode(A[r * lda + k]);
            for (int64_t j = 0; j < N; ++j) {
#if ORACLE_MUTANT == 5
                double b = bf16_decode(K == N ? B[j * ldb + k] : B[k * ldb + j]);
#else
                double b = bf16_decode(B[k * ldb + j]);
#endif
                c[j] += a * b;
            }
        }
    }
}

/* dA[i, :] = sum_n dC[i, n] * B[:, n]  i.e. dA = dC . B^T, for dC [M, N], B [K, N]. */
void oracle_gemm_da(const uint16_t* dC, int64_t M, int64_t N, int64_t lddc,
                    const uint16_t* B, int64_t K, int64_t ldb,
                    const int64_t* rows, int64_t n_rows, double* dA /* [count, K] */,
                    int n_threads) {
    int64_t count = rows ? n_rows : M;
    set_threads(n_threads);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        int64_t r = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
#if ORACLE_MUTANT == 6
                acc += bf16_decode(dC[r * lddc + n]) *
                       bf16_decode(K == N ? B[n * ldb + k] : B[k * ldb + n]);
#else
                acc += bf16_decode(dC[r * lddc + n]) * bf16_decode(B[k * ldb + n]);
#endif
            }
            dA[i * K + k] = acc;
        }
    }
}

/* dB[k, :] = sum_m A[m, k] * dC[m, :]  i.e. dB = A^T . dC, for A [M, K], dC [M, N];
 * rows selects output rows k of dB. */
void oracle_gemm_db(const uint16_t* A, int64_t M, int64_t K, int64_t lda,
                    const uint16_t* dC, int64_t N, int64_t lddc,
                    const int64_t* rows, int64_t n_rows, double* dB /* [count, N] */,
                    int n_threads) {
    int64_t count = rows ? n_rows : K;
    set_threads(n_threads);
#if ORACLE_MUTANT == 7
    int64_t m_end = M > 0 ? M - 1 : 0;
#else
    int64_t m_end = M;
#endif
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        int64_t k = rows ? rows[i] : i;
        double* d = dB + i * N;
        for (int64_t j = 0; j < N; ++j) d[j] = 0.0;
        for (int64_t m = 0; m < m_end; ++m) {
            double a = bf16_decode(A[m * lda + k]);
            for (int64_t j = 0; j < N; ++j) d[j] += a * bf16_decode(dC[m * lddc + j]);
        }
    }
}
