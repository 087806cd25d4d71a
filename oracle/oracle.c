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
 *       bias_relu / bias_silu / bias_gelu   R[m,n] = act(S[m,n] + bias[n]) with
 *                 relu(x) = max(x, 0), silu(x) = x / (1 + e^-x) and
 *                 gelu(x) = x * Phi(x) = x / 2 * (1 + erf(x / sqrt 2)) (the
 *                 exact form; the guide's epilogue list, same section, names
 *                 "bias_relu", "bias_silu", "bias_gelu" without a formula)
 *       exp and erf are the C library's fp64 functions.
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
 *   oracle_gemm_mx         the block-scaled (microscaling, "MX") GEMM:
 *       R[m,n] = sum_k (a[m,k] * 2^(sa[m,k/32] - 127)) * (b[n,k] * 2^(sb[n,k/32] - 127))
 *       FlyDSL-in-PyTorch blog, section "MXFP": operands FP8 E4M3 or packed
 *       FP4 E2M1, one E8M0 scale per 32 values along the reduction axis
 *       (BlockWise1x32), fp32 accumulation, fp16/bf16 output, K a multiple of
 *       128, unit stride along K for A and B; FlyDSL prebuilt kernels guide
 *       §3.1, the MX GEMM note (per-32 E8M0 scales).  The element codes follow
 *       the OCP microscaling formats the pages name:
 *         E4M3  s eeee mmm, bias 7: (1 + m/8) 2^(e-7), subnormal (m/8) 2^-6,
 *               no infinities, s 1111 111 is NaN (the "e4m3fn" of the pages)
 *         E2M1  s ee m, bias 1: (1 + m/2) 2^(e-1), subnormal m/2
 *         E8M0  unsigned exponent: 2^(e-127), 0xFF is NaN
 *       Layouts (the pages say "packed FP4" only; this is the library's
 *       stated format): E4M3 one byte per element, [rows, K]; E2M1 two per
 *       byte along K, [rows, K/2], element k in bits 4*(k%2) .. 4*(k%2)+3
 *       (low nibble first); scales uint8 [rows, K/32].  Every product is
 *       exact in fp64.
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
 * kind 3, 4, 5: R[m,n] = relu / silu / gelu (S[m,n] + bias[n]).
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
            } else if (kind >= 3 && kind <= 5) {
                const double x = s + bf16_to_f64(bias[n]);
                R[m * N + n] = kind == 3 ? (x > 0.0 ? x : 0.0)
                               : kind == 4 ? x / (1.0 + exp(-x))
                                           : 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
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

/* ------------------------------------------------------------ MX GEMM */

/* OCP E4M3 ("fn": no infinities): s eeee mmm, exponent bias 7. */
static double e4m3_to_f64(uint8_t c)
{
    const int sgn = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7) return NAN;
    /* normal (1 + m/8) 2^(e-7) = (8 + m) 2^(e-10); subnormal (m/8) 2^-6 = m 2^-9 */
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sgn ? -v : v;
}

/* OCP E2M1: s ee m, exponent bias 1. */
static double e2m1_to_f64(uint8_t c)
{
    const int sgn = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    /* normal (1 + m/2) 2^(e-1) = (2 + m) 2^(e-2); subnormal m/2 */
    const double v = e == 0 ? 0.5 * m : ldexp(2.0 + m, e - 2);
    return sgn ? -v : v;
}

/* OCP E8M0 scale: 2^(e-127); 0xFF is NaN. */
static double e8m0_to_f64(uint8_t c) { return c == 0xFF ? NAN : ldexp(1.0, (int)c - 127); }

/* Element k of row `row` of an MX operand (fmt 0: E4M3 [rows, ld] bytes;
 * fmt 1: E2M1 packed two per byte, [rows, ld/2] bytes). */
static double mx_elem(int fmt, const uint8_t *X, int64_t ld, int64_t row, int64_t k)
{
    if (fmt == 0) return e4m3_to_f64(X[row * ld + k]);
    const uint8_t byte = X[row * (ld / 2) + k / 2];
    return e2m1_to_f64((uint8_t)((byte >> (4 * (k % 2))) & 0xF));
}

typedef struct {
    int fa, fb;
    const uint8_t *A, *SA, *B, *SB;
    double *R;
    int64_t M, N, K;
    int64_t begin, end;
} mx_job;

static void *mx_worker(void *arg)
{
    const mx_job *j = (const mx_job *)arg;
    const int64_t nb = j->K / 32;
    for (int64_t idx = j->begin; idx < j->end; ++idx) {
        const int64_t m = idx / j->N, n = idx % j->N;
        double acc = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            const double a = mx_elem(j->fa, j->A, j->K, m, k) * e8m0_to_f64(j->SA[m * nb + k / 32]);
            const double b = mx_elem(j->fb, j->B, j->K, n, k) * e8m0_to_f64(j->SB[n * nb + k / 32]);
            acc += a * b;
        }
        j->R[idx] = acc;
    }
    return NULL;
}

/* fmt_a, fmt_b: 0 = E4M3, 1 = E2M1 (packed).  A: [M, K] elements, B: [N, K]
 * elements, SA: [M, K/32], SB: [N, K/32] E8M0 codes; R [M, N] row-major.
 * Returns 0, or 2 on a bad format or size (K must be a multiple of 32). */
int oracle_gemm_mx(int fmt_a, const uint8_t *A, const uint8_t *SA, int fmt_b, const uint8_t *B,
                   const uint8_t *SB, double *R, int64_t M, int64_t N, int64_t K, int nthreads)
{
    if ((fmt_a != 0 && fmt_a != 1) || (fmt_b != 0 && fmt_b != 1) || M < 0 || N < 0 || K < 0 || K % 32)
        return 2;
    const int64_t total = M * N;
    if (total == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)total;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof *th);
    mx_job *jobs = (mx_job *)calloc((size_t)nthreads, sizeof *jobs);
    if (!th || !jobs) { free(th); free(jobs); return 3; }
    for (int t = 0; t < nthreads; ++t) {
        mx_job j = {fmt_a, fmt_b, A, SA, B, SB, R, M, N, K, total * t / nthreads, total * (t + 1) / nthreads};
        jobs[t] = j;
        if (pthread_create(&th[t], NULL, mx_worker, &jobs[t]) != 0) {
            mx_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    free(th);
    free(jobs);
    return 0;
}

/* Decoded values of MX codes, for pins: kind 0 = E4M3, 1 = E2M1 (one code
 * per byte, low nibble), 2 = E8M0. */
int oracle_mx_decode(int kind, const uint8_t *codes, double *out, int64_t n)
{
    if (kind < 0 || kind > 2 || n < 0) return 2;
    for (int64_t i = 0; i < n; ++i)
        out[i] = kind == 0 ? e4m3_to_f64(codes[i]) : kind == 1 ? e2m1_to_f64(codes[i] & 0xF) : e8m0_to_f64(codes[i]);
    return 0;
}
