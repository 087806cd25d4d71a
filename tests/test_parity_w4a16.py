"""GPU parity of gemm_w4a16 against the fp64 oracle.

The sixteen W4A16 decode shapes are compared element by element at full
size; prefill token counts on sampled rows and columns.
The oracle is exact (fp64, unrounded dequantised weights); the library may
round each dequantised weight to bf16 (relative error <= 2^-9), well inside
the tolerance |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).  With unit (or
power-of-two) scales and integer activations every step is exact, so those
cases must match bit for bit.
"""
import numpy as np
import pytest

import oracle
from dense_bit_weight_gb300 import synth
from gpu_helpers import assert_close, assert_exact, dev_bf16, dev_raw, host_bits, sample_rows

pytestmark = pytest.mark.gpu

VARIANTS = ["gemv", "skinny", "prefill", "register", "fragment", "groupwise", "pair", "band"]


@pytest.fixture(scope="module")
def g():
    import torch
    from dense_bit_weight_gb300 import gemm
    torch.cuda.init()
    yield gemm
    assert gemm.gemm_last_device_error() == 0


def runnable(g, M, N, K, group, variant):
    try:
        p = g.gemm_w4a16_plan(M, N, K, group, variant)
    except g.GemmError:
        return False
    return not (p["variant"] == 1 and M > 64)


def operands(M, N, K, group, seed, kind):
    Bq, S, Z = synth.w4a16_operands(N, K, group, seed)
    if kind == "int":
        A = synth.bf16_int_uniform((M, K), -4, 4, seed, synth.STREAM_A_INT)
        # s = 2^-4 exactly: (q - z) * s and the whole sum stay exact in fp32
        S = np.full_like(S, 0x3D80)
    else:
        A = synth.bf16_normal((M, K), 1.0, seed, synth.STREAM_A)
    return A, Bq, S, Z


def run(g, A, Bq, S, Z, group, variant="auto"):
    C = g.gemm_w4a16(dev_bf16(A), dev_raw(Bq), dev_bf16(S), dev_raw(Z), group, variant=variant)
    return host_bits(C)


SMALL = [(1, 8, 128, 32), (1, 64, 256, 64), (2, 136, 384, 128), (3, 520, 1024, 32),
         (4, 1000, 2048, 128), (8, 264, 640, 128), (16, 136, 512, 64), (17, 4104, 256, 128),
         (64, 512, 1024, 128), (128, 392, 1280, 128), (129, 136, 512, 32),
         # K % 64 == 32: the last 64-k sub-tile is half past K (its second group is absent)
         (16, 264, 608, 32), (40, 136, 4128, 32),
         # more than 128 tokens: several token tiles per weight tile
         (300, 520, 1024, 128), (1000, 264, 2048, 64), (257, 4104, 256, 32)]


@pytest.mark.parametrize("M,N,K,group", SMALL)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_small_shapes(g, M, N, K, group, variant, kind):
    if not runnable(g, M, N, K, group, variant):
        pytest.skip(f"{variant} does not run this shape")
    A, Bq, S, Z = operands(M, N, K, group, seed=M + N, kind=kind)
    C = run(g, A, Bq, S, Z, group, variant)
    ref = oracle.gemm_w4a16(A, Bq, S, Z, group)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"{variant} {M}x{N}x{K}/{group}")


# The band kernel (M <= 8): the whole band requested at once (four stages)
# and the eight-slot ring (long K), K not a multiple of 256 (one 2-D copy per
# box, the last one half past K), fewer than four boxes, 48-row bands, the
# three group sizes.
W4_BAND = [(1, 7168, 5120, 128), (8, 5120, 17408, 128), (8, 5120, 5120, 64), (5, 1000, 2080, 32),
           (1, 152, 128, 128), (3, 7296, 1024, 128), (7, 4104, 3072, 32)]


@pytest.mark.parametrize("M,N,K,group", W4_BAND)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_band(g, M, N, K, group, kind):
    assert g.gemm_w4a16_plan(M, N, K, group, "band")["variant"] == 10
    A, Bq, S, Z = operands(M, N, K, group, seed=3 * M + N, kind=kind)
    C = run(g, A, Bq, S, Z, group, "band")
    ref = oracle.gemm_w4a16(A, Bq, S, Z, group)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"band {M}x{N}x{K}/{group}")


def test_deterministic(g):
    A, Bq, S, Z = operands(16, 5120, 5120, 128, 1, "normal")
    assert np.array_equal(run(g, A, Bq, S, Z, 128), run(g, A, Bq, S, Z, 128))


W4 = [(M, N, K) for M in (1, 16, 64, 128)
      for (N, K) in ((7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408))]
# prefill-size token counts (several 128-token tiles per weight tile)
W4 += [(512, 7168, 5120), (2048, 5120, 17408), (4096, 34816, 5120)]


@pytest.mark.parametrize("M,N,K", W4)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_full_size_w4a16(g, M, N, K, kind):
    # the sixteen decode shapes: every element; prefill token counts: sampled
    # rows and columns (up to 0.7 TMAC of fp64 work each otherwise)
    group = 128
    A, Bq, S, Z = operands(M, N, K, group, 0, kind)
    C = run(g, A, Bq, S, Z, group)
    if M <= 128:
        ref = oracle.gemm_w4a16(A, Bq, S, Z, group)
        (assert_exact if kind == "int" else assert_close)(C, ref, what=f"{M}x{N}x{K}")
        return
    rows = sample_rows(M, 2, seed=N)
    cols = sample_rows(N, 3, seed=K)
    ref_r = oracle.gemm_w4a16(A[rows], Bq, S, Z, group)
    ref_c = oracle.gemm_w4a16(A, Bq[cols], S[cols], Z[cols], group)
    if kind == "int":
        assert_exact(C[rows], ref_r, what="rows")
        assert_exact(C[:, cols], ref_c, what="cols")
    else:
        rms = float(np.sqrt(np.mean(np.concatenate([ref_r.ravel(), ref_c.ravel()]) ** 2)))
        assert_close(C[rows], ref_r, rms, what="rows")
        assert_close(C[:, cols], ref_c, rms, what="cols")
