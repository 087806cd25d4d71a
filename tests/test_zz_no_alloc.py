"""gemm_bf16_noalloc, the entry point for callers that cannot allocate.

Callers whose own allocator already holds the device memory, and loops that
cannot absorb the device-wide synchronisation of cudaMalloc/cudaFree, use this
call; it takes its split-K scratch from fixed device arrays instead of
allocating.  The test calls it through the C ABI twice in a row on each shape
and checks both results against the fp64 oracle (bit for bit on integer
inputs, |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref) on N(0,1) inputs) and
against the allocating entry point gemm_bf16 within the same tolerance.
Shapes cover the GEMV path, the band kernel, cluster split-K (skinny), the skinny kernel's
stream-K schedule with more CTAs than the fixed partials allow, prefill on
CTA pairs, and stream-K prefill that must run on fewer CTAs.

This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, assert_exact, bf16_inputs, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

# (M, N, K): GEMV, the band kernel (no scratch), cluster split-K, skinny
# stream-K over 320 weight tiles of 128 columns (its 152 partial writers need
# more than the fixed 16 MiB: 128 share the units), prefill on CTA pairs (no
# scratch), stream-K prefill on 15 tiles (64 CTAs), and 4096^3 on CTA pairs.
SHAPES = [(1, 4096, 4096), (8, 6144, 4096), (16, 4096, 4096), (128, 40960, 512), (1024, 4096, 4096),
          (300, 1200, 2056), (4096, 4096, 4096)]


def call_noalloc(g, dA, dB, C, M, N, K):
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    return g.lib.gemm_bf16_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K, N,
                                   ctypes.c_void_p(stream))


@pytest.mark.parametrize("kind", ["normal", "int"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_noalloc_matches_oracle_and_allocating_entry_point(M, N, K, kind):
    import torch
    from dense_bit_weight_gb300 import gemm as g
    A, B = bf16_inputs(M, N, K, seed=17, kind=kind)
    dA, dB = dev_bf16(A), dev_bf16(B)
    want = oracle.gemm_bf16(A, B)
    ref_alloc = oracle.bf16_bits_to_f64(host_bits(g.gemm_bf16(dA, dB)))
    free_after_first = None
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        if call == 1:
            free_after_first = torch.cuda.mem_get_info()[0]
        rc = call_noalloc(g, dA, dB, C, M, N, K)
        assert rc == 0, g.gemm_status_string(rc)
        torch.cuda.synchronize()
        got = host_bits(C)
        if kind == "int":
            assert_exact(got, want, what=f"noalloc call {call} {M}x{N}x{K}")
        else:
            assert_close(got, want, what=f"noalloc call {call} {M}x{N}x{K}")
        ok, _ = oracle.within_tolerance(oracle.bf16_bits_to_f64(got), ref_alloc)
        assert ok.all(), f"call {call}: {int((~ok).sum())} of {ok.size} differ from gemm_bf16"
    # the second call allocated nothing on the device
    assert torch.cuda.mem_get_info()[0] == free_after_first
    assert g.gemm_bf16_noalloc_last_error() == 0


def test_skinny_stream_k_case_has_more_ctas_than_the_scratch_holds():
    # the (128, 40960, 512) case above: 320 weight tiles are more than two per
    # SM, so the skinny kernel runs stream-K on every SM; 152 writers of two
    # 128 x 128 fp32 partials each exceed the fixed 16 MiB (128 fit)
    from dense_bit_weight_gb300 import gemm as g
    p = g.gemm_bf16_plan(128, 40960, 512)
    assert p["variant_name"] == "skinny" and p["tile_m"] == 128
    tiles = 40960 // 128
    assert tiles > 2 * 152 and p["grid"] > 128


@pytest.mark.parametrize("M,N,K", [(16, 512, 512), (300, 1200, 2056)])
def test_noalloc_forced_timeout_is_reported_and_recoverable(M, N, K):
    import torch
    from dense_bit_weight_gb300 import gemm as g
    A, B = bf16_inputs(M, N, K, seed=5)
    dA, dB = dev_bf16(A), dev_bf16(B)
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert g.gemm_bf16_noalloc_last_error() == 0
    g.gemm_debug_inject_timeout(True)
    try:
        assert call_noalloc(g, dA, dB, C, M, N, K) == 0
        torch.cuda.synchronize()
    finally:
        g.gemm_debug_inject_timeout(False)
    assert g.gemm_bf16_noalloc_last_error() == 7     # GEMM_ERR_DEVICE_TIMEOUT
    assert g.gemm_bf16_noalloc_last_error() == 0     # reading clears it
    assert g.gemm_last_device_error() == 0           # the allocating entry point's word is untouched
    assert call_noalloc(g, dA, dB, C, M, N, K) == 0
    torch.cuda.synchronize()
    assert_close(host_bits(C), oracle.gemm_bf16(A, B), what=f"noalloc after timeout {M}x{N}x{K}")
    assert g.gemm_bf16_noalloc_last_error() == 0


def test_noalloc_rejects_bad_arguments_without_launch():
    from dense_bit_weight_gb300 import gemm as g
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 0, 4, 16, 32, 32, 32, 16) == 1     # C NULL
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 1 << 23, 4, 16, 12, 16, 16, 16) == 2
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 1 << 23, 4, 16, 32, 24, 32, 16) == 3
    assert g.gemm_bf16_noalloc_ptr((1 << 20) + 2, 1 << 22, 1 << 23, 4, 16, 32, 32, 32, 16) == 4
