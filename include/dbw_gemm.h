/*
 * dbw_gemm.h -- C ABI of the GB300 projection-GEMM library (libdbw_gemm.so).
 *
 * The operation is the transformer projection
 *
 *     C[M,N] = A[M,K] . B[N,K]^T
 *
 * with A and B stored K-contiguous ("NT"), bf16 inputs, fp32 accumulation and
 * bf16 output (round to nearest, ties to even).  Sources: FlyDSL prebuilt
 * kernels guide, §3.1 "Preshuffle GEMM" (C = A @ B^T with B stored [N,K], M a
 * run-time argument); FlyDSL-in-PyTorch blog (aixai.ru), sections "Dense GEMM"
 * (bf16 NT shapes) and "MXFP" (unit stride along K for A and B, fp32
 * accumulation, bf16 output).  The 4-bit-weight variant is the W4A16 (AWQ)
 * decode GEMM of the hk-dsl PyPI page, section "Results".
 *
 * Conventions shared by every entry point
 *   - All matrix pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them beyond the call's stream work.
 *   - Sizes and leading dimensions are int64_t and counted in ELEMENTS.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.  Results are
 *     visible to later work on the same stream.
 *   - A precondition failure returns an error code and enqueues nothing.
 *     There is no fallback of any kind: an unsupported input is an error.
 *   - The library owns only lazily created per-device internals (the device
 *     error word and the split-K workspace), created on the first call on each
 *     device and released by gemm_shutdown().  The first call on a device
 *     (and the first split-K call on a stream) must not happen inside CUDA
 *     stream capture, because it allocates.
 *   - Determinism: identical inputs give bitwise identical outputs; K-split
 *     partial sums are added in a fixed order, with no floating-point atomics.
 *   - The device must be compute capability 10.3 (GB300, sm_103a).
 */
#ifndef DBW_GEMM_H
#define DBW_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_NULL = 1,           /* a required pointer is NULL                     */
    GEMM_ERR_SHAPE = 2,          /* negative size, K % 8 != 0, or size too large   */
    GEMM_ERR_LD = 3,             /* leading dimension < row length or not % 8      */
    GEMM_ERR_ALIGN = 4,          /* a base pointer is not 16-byte aligned          */
    GEMM_ERR_GROUP = 5,          /* W4A16 group not in {32,64,128} or K % group    */
    GEMM_ERR_CUDA = 6,           /* a CUDA runtime call or launch failed           */
    GEMM_ERR_DEVICE_TIMEOUT = 7, /* a kernel's bounded wait expired (see below)    */
    GEMM_ERR_ARCH = 8,           /* current device is not compute capability 10.3  */
    GEMM_ERR_ALIAS = 9,          /* C overlaps an input                            */
    GEMM_ERR_VARIANT = 10,       /* a forced variant cannot run this shape         */
    GEMM_ERR_EPILOGUE = 11       /* unknown epilogue, or bias missing / not used   */
} gemm_status;

/* Kernel variants (what gemm_*_plan reports and gemm_*_ex may force). */
typedef enum {
    GEMM_VARIANT_AUTO = 0,
    GEMM_VARIANT_GEMV = 1,       /* CUDA-core weight streaming, small M            */
    GEMM_VARIANT_SKINNY = 2,     /* tcgen05, weights as the MMA M side (swap AB)   */
    GEMM_VARIANT_PREFILL = 3,    /* tcgen05, persistent warp-specialised tiles     */
                                 /* (also decode whose weight rows fill one wave   */
                                 /* of 176-256-row tiles: no K split)              */
    GEMM_VARIANT_ZERO = 4,       /* K == 0: C is the empty sum, written as zeros   */
    GEMM_VARIANT_REGISTER = 5,   /* W4A16, M <= 32: weights dequantised into       */
                                 /* registers for warp-level MMAs (mma.sync)       */
    GEMM_VARIANT_FRAGMENT = 6,   /* W4A16, M <= 16: weights streamed by TMA and    */
                                 /* dequantised into mma.sync fragments            */
    GEMM_VARIANT_GROUPWISE = 7,  /* W4A16: exact 128 + q weights in tensor memory, */
                                 /* one tcgen05 accumulator per quantisation       */
                                 /* group, scale and zero applied per group        */
    GEMM_VARIANT_BLOCK_SCALED = 8, /* MX: block-scaled tcgen05 MMAs (gemm_mxfp*)   */
    GEMM_VARIANT_PAIR = 9,       /* bf16 prefill on CTA pairs: 256 x 256 tiles,    */
                                 /* tcgen05.mma.cta_group::2                       */
    GEMM_VARIANT_BAND = 10       /* decode on bands of weight rows: each SM takes  */
                                 /* at most 64 rows over all of K, TMA copies into */
                                 /* warp-level MMAs (no K split, no workspace);    */
                                 /* bf16 M <= 32, W4A16 M <= 8                     */
} gemm_variant;

typedef struct {
    int variant;   /* gemm_variant chosen                                         */
    int kernels;   /* kernel launches one call makes                              */
    int grid;      /* CTAs of the main kernel                                     */
    int split;     /* K splits per output tile (1 = none)                         */
    int tile_m;    /* output rows (M) per tile                                    */
    int tile_n;    /* output columns (N) per tile                                 */
    int stages;    /* shared-memory pipeline stages (0 for CUDA-core kernels)     */
    int reserved;
} gemm_plan;

/*
 * gemm_bf16 -- C = A . B^T, bf16 in / fp32 accumulate / bf16 out.
 *
 *   A   [M,K] bf16, row m at A + m*lda            (read only)
 *   B   [N,K] bf16, row n at B + n*ldb            (read only; the weights)
 *   C   [M,N] bf16, row m at C + m*ldc            (written; must not overlap A, B)
 *   M, N, K >= 0, K % 8 == 0, each < 2^31.  M == 0 or N == 0: nothing to do,
 *   returns GEMM_OK.  K == 0: C is set to zero.
 *   lda >= K, ldb >= K, ldc >= N, each a multiple of 8.
 *   A, B, C 16-byte aligned (rows are then 16-byte aligned too).
 *   stream: cudaStream_t.
 * Returns gemm_status.
 */
int gemm_bf16(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * gemm_w4a16 -- C = A . W^T with group-quantised 4-bit weights
 *     W[n,k] = (q[n,k] - z[n, k/group]) * s[n, k/group].
 *
 *   A       [M,K] bf16, dense (row m at A + m*K)
 *   Bq      [N,K/8] int32, dense: q[n,k] = bits 4*(k%8) .. 4*(k%8)+3 of
 *           Bq[n*(K/8) + k/8] (eight unsigned nibbles per word, low nibble
 *           first, sequential along K)
 *   scales  [N,K/group] bf16, dense
 *   zeros   [N,K/group] uint8, dense, values 0..15 (the 4-bit zero point)
 *   C       [M,N] bf16, dense (row m at C + m*N); must not overlap any input
 *   group in {32, 64, 128}; K % group == 0; K % 8 == 0; N % 8 == 0.
 *   A, Bq, C 16-byte aligned; scales 2-byte aligned.
 * The dequantised weight may be rounded to bf16 before it is multiplied
 * (relative error <= 2^-9 per weight); accumulation is fp32.
 * Returns gemm_status.
 */
int gemm_w4a16(const void *A, const void *Bq, const void *scales, const void *zeros, void *C,
               int64_t M, int64_t N, int64_t K, int64_t group, void *stream);

/*
 * gemm_bf16_fused -- gemm_bf16 with the epilogue fused into the GEMM's store.
 * The FlyDSL prebuilt-kernels guide (section 3.1, Preshuffle GEMM, the
 * `epilogue` parameter) fuses a bias and an activation into the GEMM; the
 * hk-dsl PyPI page lists a fused SiLU-mul for the gated MLP.  The epilogue is
 * applied in fp32 to the complete K sum, and the result is rounded to bf16
 * once (nearest, ties to even).
 *
 *   GEMM_EPI_NONE      C[m,n] = sum_k A[m,k] B[n,k]                (as gemm_bf16)
 *   GEMM_EPI_BIAS      C[m,n] = sum_k A[m,k] B[n,k] + bias[n]
 *                      bias: bf16 [N], 2-byte aligned, device memory.
 *   GEMM_EPI_SILU_MUL  B is the fused gate/up projection with 2N rows: gate
 *                      rows 0..N-1, then up rows N..2N-1 (row j at B + j*ldb).
 *                      g = sum_k A[m,k] B[n,k], u = sum_k A[m,k] B[N+n,k],
 *                      C[m,n] = silu(g) * u, silu(x) = x / (1 + exp(-x)).
 *                      C is [M, N]; bias must be NULL.
 *   GEMM_EPI_BIAS_RELU C[m,n] = relu(x), x = sum_k A[m,k] B[n,k] + bias[n],
 *   GEMM_EPI_BIAS_SILU relu(x) = max(x, 0), silu(x) = x / (1 + exp(-x)),
 *   GEMM_EPI_BIAS_GELU gelu(x) = x/2 (1 + erf(x / sqrt 2)) (the exact form);
 *                      bias as for GEMM_EPI_BIAS (the guide's "bias_relu",
 *                      "bias_silu", "bias_gelu").
 *
 * Sizes, leading dimensions, alignment and errors as for gemm_bf16 (N counts
 * the columns of C; B spans 2N rows for GEMM_EPI_SILU_MUL).  An unknown
 * epilogue, or a bias that is NULL for a bias epilogue or not NULL otherwise,
 * returns GEMM_ERR_EPILOGUE; C overlapping bias returns GEMM_ERR_ALIAS.
 * gemm_bf16_fused_ex forces a kernel family like gemm_bf16_ex.
 */
typedef enum {
    GEMM_EPI_NONE = 0,
    GEMM_EPI_BIAS = 1,
    GEMM_EPI_SILU_MUL = 2,
    GEMM_EPI_BIAS_RELU = 3,
    GEMM_EPI_BIAS_SILU = 4,
    GEMM_EPI_BIAS_GELU = 5
} gemm_epilogue;

int gemm_bf16_fused(const void *A, const void *B, const void *bias, void *C, int64_t M, int64_t N,
                    int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void *stream);
int gemm_bf16_fused_ex(const void *A, const void *B, const void *bias, void *C, int64_t M, int64_t N,
                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void *stream,
                       int variant);

/*
 * gemm_bf16_grouped -- the grouped (mixture-of-experts) GEMM.  The FlyDSL
 * PyTorch blog (section "Grouped GEMM: MoE with uneven load") stacks the
 * tokens routed to G experts into one activation matrix, keeps the experts'
 * weights grouped, and marks each expert's rows with offsets; one persistent
 * launch walks the tiles of all experts, so an expert with no tokens costs
 * nothing.
 *
 *   A     [M, K] bf16 (row m at A + m*lda): expert g's tokens are the rows
 *         ends[g-1] .. ends[g]-1 (ends[-1] = 0).
 *   B     [G, N, K] bf16: expert g's weights are the rows g*N .. g*N+N-1
 *         (row j at B + j*ldb).  (The blog's B[G, K, N] is the logical shape;
 *         here every expert is stored K-contiguous like gemm_bf16's B.)
 *   C     [M, N] bf16 (row m at C + m*ldc): C[m,:] = A[m,:] . B_g^T for the
 *         expert g owning row m; rows at or past ends[G-1] are not written.
 *   ends  int32 [G] device memory, 4-byte aligned: cumulative row ends,
 *         normally non-decreasing and <= M.  It may be written by the
 *         previous kernel on the stream (a router); the kernel reads it after
 *         that kernel completes.  Out-of-range values are clamped (each end to
 *         at least the previous one and at most M), so they never address
 *         outside A or C.
 * 1 <= G <= 1024, K >= 8; other sizes, leading dimensions and alignment as
 * gemm_bf16 (K == 0 returns GEMM_ERR_SHAPE).  Accumulation fp32, one bf16
 * rounding.  Runs on `stream` with no host synchronisation.
 */
int gemm_bf16_grouped(const void *A, const void *B, void *C, const void *ends, int64_t G, int64_t M,
                      int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * gemm_bf16_noalloc -- gemm_bf16 for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this is a property of the
 * library, not of the method.)
 *
 * gemm_bf16 lazily allocates its device error word and, for split-K
 * launches, a per-stream workspace.  Some callers cannot let a library call
 * cudaMalloc: a program whose own caching allocator already holds the device
 * memory budget (a library allocation would fail or fragment it), or a
 * latency-critical loop that cannot afford the implicit device
 * synchronisation of cudaMalloc/cudaFree.  They call this instead.
 * Arguments, layouts, preconditions and results are those of gemm_bf16; it
 * allocates nothing.
 *
 *   - Scratch: split-K partial tiles and per-tile counters live in fixed
 *     file-scope device arrays of the library: 16 MiB of fp32 partials and
 *     16384 counters.  Every GPU that loads the library holds them until the
 *     process exits.  When a split-K plan would need more partials than fit,
 *     fewer CTAs share the split work (full waves of whole tiles still run on
 *     every SM); a split plan with more than 16384 output tiles is rejected
 *     with GEMM_ERR_SHAPE (the current planner never splits that many tiles).
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the arrays' device addresses (cudaGetSymbolAddress).
 *   - Sharing: all calls on a device share the arrays, which keep the last
 *     call's contents.  The counters are cleared on the stream at the start
 *     of each split-K call.  Calls that overlap on the GPU (different streams
 *     without ordering between them) race on the scratch and give undefined
 *     results; order them.
 *   - Watchdog: its kernels' bounded waits end them cleanly; an expiry is
 *     recorded in a word of this entry point's own, which
 *     gemm_bf16_noalloc_last_error() reads (not gemm_last_device_error()).
 * Returns gemm_status.
 */
int gemm_bf16_noalloc(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, void *stream);

/*
 * gemm_bf16_noalloc_last_error -- the watchdog word of gemm_bf16_noalloc on
 * the current device: GEMM_ERR_DEVICE_TIMEOUT when one of its kernels' bounded
 * waits expired since the last read (C of that call is then unspecified),
 * GEMM_OK otherwise.  Reading clears it.  Call after synchronising the
 * stream; it copies one int each way (cudaMemcpyFromSymbol/ToSymbol, which
 * allocate nothing and synchronise with the legacy default stream).  After a
 * timeout the next split-K call clears the counters itself.
 */
int gemm_bf16_noalloc_last_error(void);

/*
 * gemm_mxfp8 / gemm_mxfp4 -- the block-scaled ("microscaling", MX) GEMM
 *
 *     C[m,n] = sum_k (a[m,k] * 2^(SA[m,k/32] - 127)) * (b[n,k] * 2^(SB[n,k/32] - 127))
 *
 * FlyDSL-in-PyTorch blog, section "MXFP": FP8 E4M3 or packed FP4 E2M1
 * operands, one E8M0 scale per 32 values along the reduction axis, fp32
 * accumulation, bf16 output, K a multiple of 128, unit stride along K for A
 * and B ("NT"); FlyDSL prebuilt kernels guide §3.1, the MX GEMM note.  The
 * element formats are the OCP microscaling ones: E4M3 (s eeee mmm, bias 7, no
 * infinities, 0x7F/0xFF NaN), E2M1 (s ee m, bias 1), E8M0 (2^(e - 127),
 * 0xFF NaN).  The scales are applied inside the tensor-core MMA.
 *
 *   A    gemm_mxfp8: E4M3 codes uint8 [M, K], dense.
 *        gemm_mxfp4: packed E2M1 uint8 [M, K/2], dense; element k is bits
 *        4*(k%2) .. 4*(k%2)+3 of byte k/2 (low nibble first).
 *   SA   E8M0 codes uint8 [M, K/32], dense (row m's block j at SA + m*(K/32) + j)
 *   B    as A, [N, K] or [N, K/2] (the weights)
 *   SB   E8M0 codes uint8 [N, K/32], dense
 *   C    [M, N] bf16, dense (row m at C + m*N); must not overlap any input
 *   M, N, K >= 0, K % 128 == 0, N % 8 == 0, each < 2^31.  M == 0 or N == 0:
 *   nothing to do.  K == 0: C is set to zero.
 *   A, B, C 16-byte aligned; SA, SB 4-byte aligned.  Device memory.
 * Inputs are finite (NaN codes are out of scope).  The library keeps a
 * rearranged copy of the scales in its per-stream workspace, so the call
 * allocates on first use like gemm_bf16.  Returns gemm_status.
 */
int gemm_mxfp8(const void *A, const void *SA, const void *B, const void *SB, void *C, int64_t M, int64_t N,
               int64_t K, void *stream);
int gemm_mxfp4(const void *A, const void *SA, const void *B, const void *SB, void *C, int64_t M, int64_t N,
               int64_t K, void *stream);
/* The plan of gemm_mxfp8 (fmt 0) or gemm_mxfp4 (fmt 1) with these sizes. */
int gemm_mx_plan(int64_t M, int64_t N, int64_t K, int fmt, int num_sms, gemm_plan *out);

/*
 * gemm_bf16_ex / gemm_w4a16_ex -- as above, but `variant` may force a kernel
 * family (GEMM_VARIANT_AUTO picks as the plain call does).  A forced variant
 * that cannot run the shape returns GEMM_ERR_VARIANT and enqueues nothing.
 * Meant for tests and measurements that need a specific kernel.
 */
int gemm_bf16_ex(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldc, void *stream, int variant);
int gemm_w4a16_ex(const void *A, const void *Bq, const void *scales, const void *zeros,
                  void *C, int64_t M, int64_t N, int64_t K, int64_t group, void *stream,
                  int variant);

/*
 * gemm_bf16_plan / gemm_w4a16_plan -- the launch plan a call with these sizes
 * would use, without launching anything.  num_sms > 0 plans for that many
 * SMs (host-only, no GPU needed); num_sms == 0 queries the current device.
 * Returns a gemm_status for the sizes (pointers are not checked).
 */
int gemm_bf16_plan(int64_t M, int64_t N, int64_t K, int variant, int num_sms, gemm_plan *out);
/* The plan of gemm_bf16_fused_ex with these sizes (N = columns of C; the
 * SiLU-mul epilogue multiplies 2N weight rows); GEMM_ERR_EPILOGUE for an
 * unknown epilogue. */
int gemm_bf16_fused_plan(int64_t M, int64_t N, int64_t K, int epilogue, int variant, int num_sms,
                         gemm_plan *out);
int gemm_w4a16_plan(int64_t M, int64_t N, int64_t K, int64_t group, int variant, int num_sms,
                    gemm_plan *out);

/*
 * gemm_last_device_error -- the device error word of the current device.
 * Every wait inside the tcgen05 kernels is bounded (about a second); on
 * expiry the kernel records GEMM_ERR_DEVICE_TIMEOUT here, drains its own
 * copies, frees its tensor memory and returns, so the context stays usable
 * and C holds unspecified values.  Call after synchronising the stream.
 * Reading the word clears it.  Returns GEMM_OK when nothing was recorded.
 * After a timeout, call gemm_shutdown() before further calls so the split-K
 * workspace is rebuilt from zero.
 */
int gemm_last_device_error(void);

/*
 * gemm_debug_inject_timeout -- TEST HOOK.  While enabled (non-zero), the
 * tcgen05 kernels' producer issues no tile copies, so the MMA issuer's bounded
 * wait on the first stage expires after about a second; the kernel records
 * GEMM_ERR_DEVICE_TIMEOUT in the device error word and exits cleanly (C is
 * left unspecified).  Lets a test exercise the watchdog without faulting or
 * hanging the GPU.  Process-wide; returns the previous setting.
 */
int gemm_debug_inject_timeout(int enable);

/* A static, human-readable name for a gemm_status value. */
const char *gemm_status_string(int status);

/*
 * gemm_shutdown -- synchronise every device the library has used and free
 * its internals (error words, split-K workspaces).  Later calls recreate them.
 */
void gemm_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* DBW_GEMM_H */
