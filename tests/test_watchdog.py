"""The TMA-fed kernels' bounded waits: a forced stall must end in a recorded
GEMM_ERR_DEVICE_TIMEOUT and a clean exit, leaving the context usable.

The stall is a test hook (gemm_debug_inject_timeout): the producer issues no
copies, so the MMA issuer's wait on the first stage runs out after about a
second.  Nothing faults or traps; the GPU stays usable, which the test checks
by running the same GEMM correctly afterwards.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, bf16_inputs, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant,M", [("skinny", 16), ("prefill", 256), ("pair", 512), ("band", 8)])
def test_forced_timeout_is_reported_and_recoverable(variant, M):
    import torch
    from dense_bit_weight_gb300 import gemm as g
    N, K = 512, 512
    A, B = bf16_inputs(M, N, K, seed=5)
    dA, dB = dev_bf16(A), dev_bf16(B)
    assert g.gemm_last_device_error() == 0
    g.gemm_debug_inject_timeout(True)
    try:
        g.gemm_bf16(dA, dB, variant=variant)
        torch.cuda.synchronize()
    finally:
        g.gemm_debug_inject_timeout(False)
    assert g.gemm_last_device_error() == 7          # GEMM_ERR_DEVICE_TIMEOUT
    assert g.gemm_last_device_error() == 0          # reading clears it
    g.gemm_shutdown()
    C = g.gemm_bf16(dA, dB, variant=variant)
    torch.cuda.synchronize()
    assert_close(host_bits(C), oracle.gemm_bf16(A, B), what=f"after timeout {variant}")
    assert g.gemm_last_device_error() == 0


@pytest.mark.parametrize("variant", ["skinny", "fragment", "groupwise", "band"])
def test_forced_timeout_w4a16(variant):
    import torch
    from dense_bit_weight_gb300 import gemm as g, synth
    from gpu_helpers import dev_raw
    M, N, K, group = (8 if variant == "band" else 16), 512, 1024, 128
    A = synth.bf16_normal((M, K), 1.0, 3, synth.STREAM_A)
    Bq, S, Z = synth.w4a16_operands(N, K, group, 3)
    args = (dev_bf16(A), dev_raw(Bq), dev_bf16(S), dev_raw(Z), group)
    g.gemm_debug_inject_timeout(True)
    try:
        g.gemm_w4a16(*args, variant=variant)
        torch.cuda.synchronize()
    finally:
        g.gemm_debug_inject_timeout(False)
    assert g.gemm_last_device_error() == 7
    g.gemm_shutdown()
    C = g.gemm_w4a16(*args, variant=variant)
    torch.cuda.synchronize()
    assert_close(host_bits(C), oracle.gemm_w4a16(A, Bq, S, Z, group), what="w4a16 after timeout")
    assert g.gemm_last_device_error() == 0


def test_forced_timeout_mx():
    import torch
    from dense_bit_weight_gb300 import gemm as g, synth
    M, N, K = 256, 512, 512
    A, SA = synth.mx_operands(M, K, "e4m3", seed=1, role="a")
    B, SB = synth.mx_operands(N, K, "e4m3", seed=2, role="b")
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    args = (dev(A), dev(SA), dev(B), dev(SB))
    g.gemm_debug_inject_timeout(True)
    try:
        g.gemm_mx(*args, "e4m3")
        torch.cuda.synchronize()
    finally:
        g.gemm_debug_inject_timeout(False)
    assert g.gemm_last_device_error() == 7
    g.gemm_shutdown()
    C = g.gemm_mx(*args, "e4m3")
    torch.cuda.synchronize()
    assert_close(host_bits(C), oracle.gemm_mx(A, SA, B, SB), what="mx after timeout")
    assert g.gemm_last_device_error() == 0
