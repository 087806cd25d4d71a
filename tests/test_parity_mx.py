"""GPU parity of the block-scaled (MX) GEMM, gemm_mxfp8 and gemm_mxfp4, against
the fp64 oracle.

Integer elements in [-4, 4] with unit scales make every product and partial
sum exact in fp32, so those cases must match bit for bit; random codes (E4M3
exponent fields 2^-3 .. 2^3, all E2M1 codes, scales 2^-3 .. 2^3) must satisfy
|out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).  Shapes cover 128- and 256-row B
tiles, whole tiles and stream-K, ragged M and N, K with a half stage at the
end (E2M1 stages are 256 values), and the pages' MXFP shapes at full size.
"""
import numpy as np
import pytest

import oracle
from dense_bit_weight_gb300 import synth
from gpu_helpers import assert_close, assert_exact, host_bits, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import torch
    from dense_bit_weight_gb300 import gemm
    torch.cuda.init()
    yield gemm
    assert gemm.gemm_last_device_error() == 0


def dev_u8(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def operands(M, N, K, fmt, kind, seed):
    A, SA = synth.mx_operands(M, K, fmt, seed=seed, role="a", kind=kind)
    B, SB = synth.mx_operands(N, K, fmt, seed=seed + 1, role="b", kind=kind)
    return A, SA, B, SB


def run(g, A, SA, B, SB, fmt):
    return host_bits(g.gemm_mx(dev_u8(A), dev_u8(SA), dev_u8(B), dev_u8(SB), fmt))


SMALL = [(128, 128, 128), (1, 8, 128), (37, 120, 384), (128, 256, 256), (200, 264, 512),
         (300, 1000, 640), (1024, 1024, 1024), (16, 4096, 2048), (513, 2056, 128)]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("kind", ["int", "random"])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_small(g, M, N, K, fmt, kind):
    A, SA, B, SB = operands(M, N, K, fmt, kind, seed=M + N + K)
    C = run(g, A, SA, B, SB, fmt)
    ref = oracle.gemm_mx(A, SA, B, SB, fmt, fmt)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"{fmt} {kind} {M}x{N}x{K}")


def test_k_zero_and_empty(g):
    import torch
    C = torch.full((4, 16), 3.0, dtype=torch.bfloat16, device="cuda")
    e = torch.empty((4, 0), dtype=torch.uint8, device="cuda")
    assert g.lib.gemm_mxfp8(e.data_ptr(), e.data_ptr(), e.data_ptr(), e.data_ptr(), C.data_ptr(), 4, 16, 0,
                            None) == 0
    torch.cuda.synchronize()
    assert not host_bits(C).any()


# the pages' MXFP shapes (32 x 4096 x 4096 for MXFP8, 32 x 14336 x 4096 for
# MXFP4) and prefill sizes: every element up to 2 GMAC, sampled rows and
# columns beyond
FULL = [(32, 4096, 4096), (32, 14336, 4096), (1024, 4096, 4096), (4096, 8192, 8192)]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("kind", ["int", "random"])
@pytest.mark.parametrize("M,N,K", FULL)
def test_full_size(g, M, N, K, fmt, kind):
    A, SA, B, SB = operands(M, N, K, fmt, kind, seed=0)
    C = run(g, A, SA, B, SB, fmt)
    if M * N * K <= 2 ** 31:
        ref = oracle.gemm_mx(A, SA, B, SB, fmt, fmt)
        (assert_exact if kind == "int" else assert_close)(C, ref, what=f"{fmt} {M}x{N}x{K}")
        return
    rows = sample_rows(M, 2, seed=N)
    cols = sample_rows(N, 2, seed=K)
    ref_r = oracle.gemm_mx(A[rows], SA[rows], B, SB, fmt, fmt)
    ref_c = oracle.gemm_mx(A, SA, B[cols], SB[cols], fmt, fmt)
    if kind == "int":
        assert_exact(C[rows], ref_r, what="rows")
        assert_exact(C[:, cols], ref_c, what="cols")
    else:
        rms = float(np.sqrt(np.mean(np.concatenate([ref_r.ravel(), ref_c.ravel()]) ** 2)))
        assert_close(C[rows], ref_r, rms, what="rows")
        assert_close(C[:, cols], ref_c, rms, what="cols")
