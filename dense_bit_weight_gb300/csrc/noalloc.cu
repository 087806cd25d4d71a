// noalloc.cu -- gemm_bf16_noalloc: the bf16 GEMM for callers that cannot
// allocate device memory.
//
// gemm_bf16 lazily cudaMalloc's a device error word and, for split-K
// (stream-K) launches, a per-stream workspace of fp32 partial tiles and
// per-tile arrival counters.  Some callers cannot let a library do that:
// programs whose caching allocator has already reserved the device's memory
// budget, and latency-critical loops where the implicit device
// synchronisation of cudaMalloc/cudaFree would stall other streams.  This
// entry point runs the same kernels with the split-K scratch taken from fixed
// arrays in this file instead.
//
// The arrays are file-scope __device__ objects, so every GPU that loads the
// library holds them (16 MiB of partials, 64 KiB of counters, one error
// word) until the process exits.  In host code their names are host-side
// stand-ins, not device addresses; the device addresses come from
// cudaGetSymbolAddress, once per device, on the first call with that device
// current.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

using namespace dbw;

constexpr int64_t kScratchFloats = int64_t(1) << 22;   // 16 MiB of fp32 partial tiles
constexpr int64_t kScratchCounters = 16384;             // per-tile arrival counters
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_scratch_partials[kScratchFloats];
static __device__ __align__(256) int g_scratch_counters[kScratchCounters];
static __device__ __align__(256) int g_scratch_error[64];   // [0]: watchdog word of this entry point

struct ScratchPtrs {
    bool ready = false;
    int sm_count = 0;
    float *partials = nullptr;
    int *counters = nullptr;
    int *error = nullptr;
};

std::mutex g_mu;
ScratchPtrs g_ptrs[kMaxDevices];

// Per-device set-up: the device addresses of the scratch arrays.  No allocation.
int scratch_for_device(ScratchPtrs **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    ScratchPtrs &s = g_ptrs[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (!(major == 10 && minor == 3)) return GEMM_ERR_ARCH;
        void *p = nullptr, *c = nullptr, *e = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch_partials) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaGetSymbolAddress(&c, g_scratch_counters) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaGetSymbolAddress(&e, g_scratch_error) != cudaSuccess) return GEMM_ERR_CUDA;
        s.partials = static_cast<float *>(p);
        s.counters = static_cast<int *>(c);
        s.error = static_cast<int *>(e);
        s.sm_count = sms;
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

bool is_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

int64_t span_bytes(int64_t rows, int64_t cols, int64_t ld) { return rows == 0 ? 0 : ((rows - 1) * ld + cols) * 2; }

}  // namespace

extern "C" int gemm_bf16_noalloc(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                                 int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    // the same preconditions as gemm_bf16
    const int64_t kMax = (int64_t(1) << 31) - 1;
    if (M < 0 || N < 0 || K < 0 || M > kMax || N > kMax || K > kMax || K % 8) return GEMM_ERR_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_NULL;
    if (ldc < N || ldc % 8 || (K > 0 && (lda < K || ldb < K || lda % 8 || ldb % 8))) return GEMM_ERR_LD;
    if (!is_aligned16(C) || (K > 0 && (!is_aligned16(A) || !is_aligned16(B)))) return GEMM_ERR_ALIGN;
    const int64_t cb = span_bytes(M, N, ldc);
    if (K > 0 && (ranges_overlap(C, cb, A, span_bytes(M, K, lda)) || ranges_overlap(C, cb, B, span_bytes(N, K, ldb))))
        return GEMM_ERR_ALIAS;

    ScratchPtrs *s = nullptr;
    int rc = scratch_for_device(&s);
    if (rc) return rc;
    Plan p;
    if (!plan_bf16(M, N, K, GEMM_VARIANT_AUTO, s->sm_count, &p)) return GEMM_ERR_SHAPE;
    const cudaStream_t st = (cudaStream_t)stream;
    LaunchCtx c{};
    c.stream = st;
    c.sm_count = s->sm_count;
    c.d_error = s->error;
    c.workspace = s->partials;
    c.counters = s->counters;
    c.ws_floats = kScratchFloats;
    c.n_counters = kScratchCounters;

    const bool umma = p.variant == GEMM_VARIANT_SKINNY || p.variant == GEMM_VARIANT_PREFILL;
    if (umma && p.mode == 1) {
        // fit the split-K partials in the fixed array.  Only the CTAs that
        // share the stream-K units write partials (two tiles' worth each):
        // when full waves of whole tiles come first, only those sharing CTAs
        // are capped and every SM still takes whole tiles; a plan that is
        // stream-K throughout runs on fewer CTAs instead.
        const int64_t per_cta = 2 * (int64_t)kUmmaBM * p.bn;
        const int64_t max_writers = kScratchFloats / per_cta;
        if (p.whole > 0 && p.sk_grid > 0) {
            if (p.sk_grid > max_writers) p.sk_grid = (int)max_writers;
        } else if (p.grid > max_writers) {
            p.grid = (int)max_writers;
        }
        int64_t R = p.variant == GEMM_VARIANT_SKINNY ? N : M, Q = p.variant == GEMM_VARIANT_SKINNY ? M : N;
        const int64_t tiles = ((R + kUmmaBM - 1) / kUmmaBM) * ((Q + p.bn - 1) / p.bn);
        if (tiles > kScratchCounters) return GEMM_ERR_SHAPE;
        // the counters must start at zero; an earlier call that timed out may have left some set
        if (cudaMemsetAsync(s->counters, 0, (size_t)tiles * sizeof(int), st) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    if (p.variant == GEMM_VARIANT_PAIR && p.mode == 1) {
        // CTA pairs: both CTAs of a sharing pair keep two 128 x 256 partials
        const int64_t per_pair = 4 * (int64_t)kUmmaBM * p.bn;
        const int64_t max_pairs = kScratchFloats / per_pair;
        if (p.sk_grid > max_pairs) p.sk_grid = (int)max_pairs;
        if (p.whole == 0) p.grid = 2 * p.sk_grid;   // stream-K throughout: only the sharing pairs run
        const int64_t counters = 2 * ((M + 255) / 256) * ((N + p.bn - 1) / p.bn);
        if (counters > kScratchCounters) return GEMM_ERR_SHAPE;
        if (cudaMemsetAsync(s->counters, 0, (size_t)counters * sizeof(int), st) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    GemmArgs a{A, B, nullptr, nullptr, C, M, N, K, lda, ldb, ldc, 0};
    cudaError_t e;
    switch (p.variant) {
    case GEMM_VARIANT_ZERO: e = launch_zero_fill(a, c); break;
    case GEMM_VARIANT_GEMV: e = launch_gemv_bf16(a, p, c); break;
    case GEMM_VARIANT_BAND: e = launch_gemv_band(a, p, c); break;
    case GEMM_VARIANT_PAIR: e = launch_umma_pair(a, p, c); break;
    default: e = launch_umma_bf16(a, p, c); break;
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

extern "C" int gemm_bf16_noalloc_last_error(void)
{
    // the word gemm_bf16_noalloc's kernels write on a bounded-wait expiry;
    // read and cleared with symbol copies, which allocate nothing
    ScratchPtrs *s = nullptr;
    int rc = scratch_for_device(&s);
    if (rc) return rc;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_scratch_error, sizeof v, 0, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_scratch_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    return v;
}
