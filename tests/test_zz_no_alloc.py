"""gemm_bf16_noalloc, the entry point for callers that cannot allocate.

Callers inside CUDA-graph capture (global mode refuses cudaMalloc), callers
whose own allocator already holds the device memory, and loops that cannot
absorb the device-wide synchronisation of cudaMalloc/cudaFree use this call;
it takes its split-K scratch from fixed device arrays instead of allocating.
The test calls it through the C ABI twice in a row on each shape and checks
both results against gemm_bf16 (the allocating entry point) within the
tolerance every parity test uses, |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).
Shapes cover the plain GEMV path, the split-K tensor-core paths (skinny and
prefill, the latter with more CTAs than the fixed partials allow, so the
call shares the work among fewer CTAs) and whole-tile prefill.

This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_helpers import bf16_inputs, dev_bf16, host_bits

pytestmark = pytest.mark.gpu

SHAPES = [(1, 4096, 4096), (16, 4096, 4096), (128, 6144, 4096), (1024, 4096, 4096),
          (300, 1200, 2056), (4096, 4096, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_noalloc_matches_allocating_entry_point(M, N, K):
    import torch
    from dense_bit_weight_gb300 import gemm as g
    A, B = bf16_inputs(M, N, K, seed=17)
    dA, dB = dev_bf16(A), dev_bf16(B)
    ref = host_bits(g.gemm_bf16(dA, dB))
    ref_f = oracle.bf16_bits_to_f64(ref)
    stream = torch.cuda.current_stream().cuda_stream
    free_after_first = None
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        if call == 1:
            free_after_first = torch.cuda.mem_get_info()[0]
        rc = g.lib.gemm_bf16_noalloc(dA.data_ptr(), dB.data_ptr(), C.data_ptr(), M, N, K, K, K, N,
                                     ctypes.c_void_p(stream))
        assert rc == 0, g.gemm_status_string(rc)
        torch.cuda.synchronize()
        out = oracle.bf16_bits_to_f64(host_bits(C))
        ok, _ = oracle.within_tolerance(out, ref_f)
        assert ok.all(), f"call {call}: {int((~ok).sum())} of {ok.size} outside tolerance"
    # the second call allocated nothing on the device
    assert torch.cuda.mem_get_info()[0] == free_after_first


def test_noalloc_rejects_bad_arguments_without_launch():
    from dense_bit_weight_gb300 import gemm as g
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 0, 4, 16, 32, 32, 32, 16) == 1     # C NULL
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 1 << 23, 4, 16, 12, 16, 16, 16) == 2
    assert g.gemm_bf16_noalloc_ptr(1 << 20, 1 << 22, 1 << 23, 4, 16, 32, 24, 32, 16) == 3
    assert g.gemm_bf16_noalloc_ptr((1 << 20) + 2, 1 << 22, 1 << 23, 4, 16, 32, 32, 32, 16) == 4
