/*
 * oracle.c -- the fp64 CPU oracle for the projection GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no source with the CUDA path.
 *
 * What it computes (plain definitions, no blocking, no fusion, no reordering):
 *
 *   oracle_gemm_bf16    R[m,n] = sum_{k<K} A[m,k] * B[n,k]
 *       The contraction C[M,N] = A[M,K] @ B[N,K]^T with A and B both stored
 *       K-contiguous ("NT" layout): FlyDSL prebuilt kernels guide, §3.1
 *       "Preshuffle GEMM" (C = A @ B^T, B is [N,K]); FlyDSL-in-PyTorch blog,
 *       section "Dense GEMM" (bf16 NT shapes) and section "MXFP" (unit stride
 *       along K for A and B; fp32 accumulation, bf16 output).
 *       The oracle accumulates in fp64 in increasing k and returns the
 *       unrounded sum.  Every bf16 x bf16 product is exact in fp64.
 *
 *   oracle_gemm_w4a16   R[m,n] = sum_{k<K} A[m,k] * (q[n,k] - z[n,k/g]) * s[n,k/g]
 *       The 4-bit-weight (AWQ-style) variant: hk-dsl (PyPI), "Results",
 *       kernels inside the engines, "W4A16 decode GEMM (AWQ)".  The pages do
 *       not spell out the dequantisation, so this follows the plain reading:
 *       q and z unsigned 4-bit values in [0,15], s a bf16 scale, one (s,z)
 *       pair per group of g consecutive k of a weight row; weight
 *       w = (q - z) * s with no further offset.
 *       Layouts (the pages are silent; this is the library's stated format):
 *         Bq     int32 [N, K/8]: q[n,k] is bits 4*(k%8) .. 4*(k%8)+3 of
 *                Bq[n, k/8] (low nibble first, sequential along K)
 *         scales bf16  [N, K/g]
 *         zeros  uint8 [N, K/g] (values 0..15)
 *       Every product A*(q-z)*s is exact in fp64 (8 + 5 + 8 significant bits).
 *
 *   oracle_round_to_bf16   fp64 -> bf16 bits, round to nearest, ties to even
 *       (the output rounding; FlyDSL prebuilt kernels guide, §2 norm kernels:
 *       "software round-to-nearest-even (RNE) pack").  Done directly from
 *       fp64, not through fp32, so there is a single rounding.
 *
 *   oracle_dequant_w4      fp64 [N,K] weights (q - z) * s, for invariant checks.
 *
 *   oracle_epilogue        the fused epilogues, applied to unrounded fp64 sums:
 *       bias      R[m,n] = S[m,n] + bias[n]   (FlyDSL prebuilt kernels guide,
 *                 section 3.1 "Preshuffle GEMM", the epilogue parameter:
 *                 "bias" and bias + activation fused into the GEMM)
 *       silu_mul  R[m,n] = silu(G[m,n]) * U[m,n], silu(x) = x / (1 + e^-x),
 *                 with G and U the gate and up halves of a fused gate/up
 *                 projection (hk-dsl PyPI page: the fused SiLU-mul kernel)
 *       exp is the C library's fp64 exp.
 *
 *   oracle_gemm_grouped    the grouped (mixture-of-experts) GEMM: expert g
 *       owns the token rows [end[g-1], end[g]) of the stacked activations
 *       A [M,K] (end[-1] = 0, end = cumulative row ends) and multiplies them
 *       by its own weights B_g [N,K] (B is [G,N,K]):
 *       R[m,n] = sum_k A[m,k] * B_g[n,k] for every m of expert g; rows of
 *       no expert are 0.  FlyDSL-in-PyTorch blog, section "Grouped GEMM: MoE
 *       with uneven load" (concatenated activations, grouped weights,
 *       offsets marking each expert's rows; empty experts own no rows).
 *
 * Threads: outputs are split into contiguous ranges of the flattened (m,n)
 * index over POSIX threads; each output is computed by exactly one thread in
 * the same k order, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* bf16 bits -> fp64, exact: the bits are the top half of an IEEE fp32. */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_hardware_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---------------------------------------------------------------- bf16 GEMM */

typedef struct {
    const uint16_t *A, *B;
    double *R;
    int64_t M, N, K, lda, ldb;
    int64_t begin, end; /* flattened output range [begin, end) */
} bf16_job;

static void *bf16_worker(void *arg)
{
    const bf16_job *j = (const bf16_job *)arg;
    for (int64_t idx = j->begin; idx < j->end; ++idx) {
        int64_t m = idx / j->N, n = idx % j->N;
        const uint16_t *a = j->A + m * j->lda;
        const uint16_t *b = j->B + n * j->ldb;
        double acc = 0.0;
        for (int64_t k = 0; k < j->K; ++k)
            acc += bf16_to_f64(a[k]) * bf16_to_f64(b[k]);
        j->R[idx] = acc;
    }
    return NULL;
}

/* R is [M,N] row-major (leading dimension N). Returns 0 on success. */
int oracle_gemm_bf16(const uint16_t *A, const uint16_t *B, double *R,
                     int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                     int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K) return 2;
    int64_t total = M * N;
    if (total == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof *th);
    bf16_job *jobs = (bf16_job *)calloc((size_t)nthreads, sizeof *jobs);
    if (!th || !jobs) { free(th); free(jobs); return 3; }
    for (int t = 0; t < nthreads; ++t) {
        bf16_job j = {A, B, R, M, N, K, lda, ldb,
                      total * t / nthreads, total * (t + 1) / nthreads};
        jobs[t] = j;
        if (pthread_create(&th[t], NULL, bf16_worker, &jobs[t]) != 0) {
            bf16_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* --------------------------------------------------------------- W4A16 GEMM */

/* The 4-bit code q[n,k] under the stated packing. */
static int nibble_at(const int32_t *Bq_row, int64_t k)
{
    uint32_t word = (uint32_t)Bq_row[k / 8];
    return (int)((word >> (4 * (k % 8))) & 0xFu);
}

typedef struct {
    const uint16_t *A;
    const int32_t *Bq;
    const uint16_t *S;
    const uint8_t *Z;
    double *R;
    int64_t M, N, K, g, lda;
    int64_t begin, end;
} w4_job;

static void *w4_worker(void *arg)
{
    const w4_job *j = (const w4_job *)arg;
    const int64_t words = j->K / 8, groups = j->K / j->g;
    for (int64_t idx = j->begin; idx < j->end; ++idx) {
        int64_t m = idx / j->N, n = idx % j->N;
        const uint16_t *a = j->A + m * j->lda;
        const int32_t *q = j->Bq + n * words;
        const uint16_t *s = j->S + n * groups;
        const uint8_t *z = j->Z + n * groups;
        double acc = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            int64_t grp = k / j->g;
            double w = (double)(nibble_at(q, k) - (int)z[grp]) * bf16_to_f64(s[grp]);
            acc += bf16_to_f64(a[k]) * w;
        }
        j->R[idx] = acc;
    }
    return NULL;
}

/* A is [M,K] with leading dimension lda; Bq/scales/zeros are dense as stated
 * above.  R is [M,N] row-major.  Returns 0 on success. */
int oracle_gemm_w4a16(const uint16_t *A, const int32_t *Bq, const uint16_t *scales,
                      const uint8_t *zeros, double *R, int64_t M, int64_t N,
                      int64_t K, int64_t group, int64_t lda, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || group <= 0 || K % 8 || K % group)
        return 2;
    int64_t total = M * N;
    if (total == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof *th);
    w4_job *jobs = (w4_job *)calloc((size_t)nthreads, sizeof *jobs);
    if (!th || !jobs) { free(th); free(jobs); return 3; }
    for (int t = 0; t < nthreads; ++t) {
        w4_job j = {A, Bq, scales, zeros, R, M, N, K, group, lda,
                    total * t / nthreads, total * (t + 1) / nthreads};
        jobs[t] = j;
        if (pthread_create(&th[t], NULL, w4_worker, &jobs[t]) != 0) {
            w4_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* W[n,k] = (q[n,k] - z[n,k/g]) * s[n,k/g] in fp64, W dense [N,K]. */
int oracle_dequant_w4(const int32_t *Bq, const uint16_t *scales, const uint8_t *zeros,
                      double *W, int64_t N, int64_t K, int64_t group)
{
    if (N < 0 || K < 0 || group <= 0 || K % 8 || K % group) return 2;
    const int64_t words = K / 8, groups = K / group;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            int64_t grp = k / group;
            W[n * K + k] = (double)(nibble_at(Bq + n * words, k) - (int)zeros[n * groups + grp]) *
                           bf16_to_f64(scales[n * groups + grp]);
        }
    return 0;
}

/* ------------------------------------------------------------ bf16 rounding */

/* Round one finite fp64 to the nearest bf16 (ties to even), return its bits.
 * bf16 keeps 8 significant bits and fp32's exponent range; its subnormal
 * spacing is 2^-133.  The value is scaled by the spacing of its binade so the
 * rounding is rint() in the default round-to-nearest-even mode. */
static uint16_t round_one(double x)
{
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    if (isinf(x)) return signbit(x) ? 0xFF80 : 0x7F80;
    int e2;
    frexp(x, &e2);            /* |x| = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;           /* |x| in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;   /* subnormal range: fixed spacing */
    double quantum = ldexp(1.0, e - 7);
    double r = rint(x / quantum) * quantum;   /* exact scaling by powers of 2 */
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)r;       /* r is a bf16 value, exactly representable */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void oracle_round_to_bf16(const double *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = round_one(x[i]);
}

/* -------------------------------------------------------------- epilogues */

/* kind 1: R[m,n] = S[m,n] + bias[n] (bias bf16 bits [N]); S is [M,N].
 * kind 2: R[m,n] = silu(S[m,n]) * U[m,n], both [M,N].
 * R may alias S.  Returns 0 on success, 2 on a bad kind or size. */
int oracle_epilogue(int kind, const double *S, const double *U, const uint16_t *bias, double *R,
                    int64_t M, int64_t N)
{
    if (M < 0 || N < 0) return 2;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            const double s = S[m * N + n];
            if (kind == 1) {
                R[m * N + n] = s + bf16_to_f64(bias[n]);
            } else if (kind == 2) {
                R[m * N + n] = s / (1.0 + exp(-s)) * U[m * N + n];
            } else {
                return 2;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------ grouped GEMM */

/* A [M,K], B [G,N,K] (expert g at B + g*N*K), R [M,N]; ends int32 [G],
 * cumulative row ends (non-decreasing, <= M).  Returns 0, or 2 on bad sizes
 * or offsets. */
int oracle_gemm_grouped(const uint16_t *A, const uint16_t *B, const int32_t *ends, double *R,
                        int64_t G, int64_t M, int64_t N, int64_t K, int nthreads)
{
    if (G < 1 || M < 0 || N < 0 || K < 0) return 2;
    memset(R, 0, (size_t)(M * N) * sizeof(double));
    int64_t start = 0;
    for (int64_t g = 0; g < G; ++g) {
        const int64_t end = ends[g];
        if (end < start || end > M) return 2;
        if (end > start) {
            const int rc = oracle_gemm_bf16(A + start * K, B + g * N * K, R + start * N, end - start, N, K, K, K,
                                            nthreads);
            if (rc) return rc;
        }
        start = end;
    }
    return 0;
}
