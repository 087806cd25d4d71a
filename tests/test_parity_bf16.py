"""GPU parity of gemm_bf16 against the fp64 oracle.

Small and ragged shapes are compared element by element, for every kernel
variant that can run the shape.  The workload shapes run at full size in the
launch configuration the bench times: every element of C is compared for the
twelve decode shapes, the five down-projection shapes and the M = 1024
prefill row; the M = 4096 and 16384 prefill shapes (1-4 TMAC each, minutes of
fp64 work on the host) are checked on sampled rows and columns the oracle
computes one by one.
Integer-valued inputs must match bit for bit; N(0,1) inputs must satisfy
|out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import assert_close, assert_exact, bf16_inputs, dev_bf16, host_bits, sample_rows

pytestmark = pytest.mark.gpu

VARIANTS = ["gemv", "skinny", "prefill", "pair", "band"]


@pytest.fixture(scope="module")
def g():
    import torch
    from dense_bit_weight_gb300 import gemm
    torch.cuda.init()
    yield gemm
    assert gemm.gemm_last_device_error() == 0


def runnable(g, M, N, K, variant):
    try:
        p = g.gemm_bf16_plan(M, N, K, variant)
    except g.GemmError:
        return False
    # one pass over the weights per group of 4 rows makes large-M GEMV slow:
    # skip it for shapes a tcgen05 variant serves
    return not (p["variant"] == 1 and M > 64)


SMALL = [(1, 8, 8), (1, 136, 24), (3, 8, 16), (4, 4104, 136), (8, 520, 64), (16, 136, 136),
         (17, 1000, 264), (33, 8, 1032), (129, 264, 72), (256, 256, 256), (255, 392, 520),
         (1000, 136, 136), (129, 4104, 8), (300, 1200, 4096),
         (8, 40960, 512)]   # skinny stream-K: 320 weight tiles, more than two per SM


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("variant", VARIANTS)
def test_small_shapes_random(g, M, N, K, variant):
    if not runnable(g, M, N, K, variant):
        pytest.skip(f"{variant} does not run {M}x{N}x{K}")
    A, B = bf16_inputs(M, N, K, seed=M + N + K)
    C = g.gemm_bf16(dev_bf16(A), dev_bf16(B), variant=variant)
    assert_close(host_bits(C), oracle.gemm_bf16(A, B), what=f"{variant} {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("variant", VARIANTS)
def test_small_shapes_integer_exact(g, M, N, K, variant):
    if not runnable(g, M, N, K, variant):
        pytest.skip(f"{variant} does not run {M}x{N}x{K}")
    A, B = bf16_inputs(M, N, K, seed=7, kind="int")
    C = g.gemm_bf16(dev_bf16(A), dev_bf16(B), variant=variant)
    assert_exact(host_bits(C), oracle.gemm_bf16(A, B), what=f"{variant} {M}x{N}x{K}")


# Prefill kernel with one token tile and the wide weight tiles the planner picks
# for it (176, 192 or 224 rows, a single wave): ragged N, K and M.  The token
# copies cover only M rows rounded up to 16; the MMA rows beyond hold stale data.
WIDE = [(100, 24536, 72, 176), (17, 24576, 136, 176), (5, 24576, 64, 176), (64, 28000, 40, 192),
        (128, 32760, 64, 224)]


@pytest.mark.parametrize("M,N,K,bn", WIDE)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_wide_single_token_tile(g, M, N, K, bn, kind):
    p = g.gemm_bf16_plan(M, N, K)
    if p["grid"] * 100 < 85 * 152 or p["tile_n"] != bn:
        pytest.skip(f"plan on this device: {p}")
    A, B = bf16_inputs(M, N, K, seed=M + K, kind=kind)
    C = g.gemm_bf16(dev_bf16(A), dev_bf16(B))
    ref = oracle.gemm_bf16(A, B)
    (assert_exact if kind == "int" else assert_close)(host_bits(C), ref, what=f"wide {bn} {M}x{N}x{K}")


# CTA pairs (256 x 256 tiles) under stream-K: a handful of tiles over every
# pair (each tile split among two to seven pairs, ragged M, N and K).
PAIR_STREAM_K = [(300, 1200, 4096), (700, 1000, 1000), (512, 4096, 1024)]


@pytest.mark.parametrize("M,N,K", PAIR_STREAM_K)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_pair_stream_k(g, M, N, K, kind):
    p = g.gemm_bf16_plan(M, N, K, "pair")
    if p["grid"] != 152:
        pytest.skip(f"plan on this device: {p}")
    assert p["split"] > 1
    A, B = bf16_inputs(M, N, K, seed=M + 3 * K, kind=kind)
    dA, dB = dev_bf16(A), dev_bf16(B)
    C = host_bits(g.gemm_bf16(dA, dB, variant="pair"))
    ref = oracle.gemm_bf16(A, B)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"pair stream-K {M}x{N}x{K}")
    # the fixup sums in a fixed order: a second call gives the same bits
    assert np.array_equal(host_bits(g.gemm_bf16(dA, dB, variant="pair")), C)


@pytest.mark.parametrize("kind", ["normal", "int"])
def test_pair_full_waves_then_split_leftovers(g, kind):
    # 96 pair tiles on 76 pairs: one wave of whole tiles, then the 20 leftover
    # tiles (columns 4864-6143 in the grouped raster) split three ways along
    # K = 4800 (75 k-blocks, a ragged last block).  Checked on every column of
    # sampled rows and on every row of sampled columns, half of them in the
    # leftover tiles.
    M, N, K = 1024, 6144, 4800
    p = g.gemm_bf16_plan(M, N, K)
    if p["grid"] != 152:
        pytest.skip(f"plan on this device: {p}")
    assert p["variant"] == 9 and p["split"] == 3
    A, B = bf16_inputs(M, N, K, seed=21, kind=kind)
    dA, dB = dev_bf16(A), dev_bf16(B)
    C = host_bits(g.gemm_bf16(dA, dB))
    rows = sample_rows(M, 4, seed=5)
    cols = np.concatenate([sample_rows(4864, 2, seed=6), 4864 + sample_rows(N - 4864, 2, seed=7)])
    ref_r = oracle.gemm_bf16(A[rows], B)
    ref_c = oracle.gemm_bf16(A, B[cols])
    if kind == "int":
        assert_exact(C[rows], ref_r, what="rows")
        assert_exact(C[:, cols], ref_c, what="cols")
    else:
        rms = float(np.sqrt(np.mean(np.concatenate([ref_r.ravel(), ref_c.ravel()]) ** 2)))
        assert_close(C[rows], ref_r, rms, what="rows")
        assert_close(C[:, cols], ref_c, rms, what="cols")
    assert np.array_equal(host_bits(g.gemm_bf16(dA, dB)), C)


# The band kernel (bf16 decode, M <= 32): K tails of half an MMA step
# (K % 16 == 8) in the first and in a later chunk, bands of exactly 64 rows,
# bands shorter than one MMA tile, 1-32 tokens, and the decode shapes at full
# size with every element compared.
BAND = [(1, 152, 8), (5, 1000, 3080), (32, 9728, 520), (17, 304, 4104), (9, 64, 2056), (31, 7000, 1024),
        (1, 6144, 4096), (8, 4096, 4096), (32, 6144, 4096), (16, 4096, 12288)]


@pytest.mark.parametrize("M,N,K", BAND)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_band(g, M, N, K, kind):
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = g.gemm_bf16_plan(M, N, K, "band")
    assert p["variant"] == 10 and p["grid"] == min(N, sms)
    A, B = bf16_inputs(M, N, K, seed=M * 7 + N + K, kind=kind)
    C = host_bits(g.gemm_bf16(dev_bf16(A), dev_bf16(B), variant="band"))
    ref = oracle.gemm_bf16(A, B)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"band {M}x{N}x{K}")


@pytest.mark.parametrize("M,K", [(5, 4096), (8, 200)])   # 3-D k-block copies / 2-D boxes (K % 64 != 0)
def test_band_leading_dimensions(g, M, K):
    # the band kernel on strided views: lda = K + 16, ldb = K + 64, ldc = N + 24
    import torch
    N = 3000
    A, B = bf16_inputs(M, N, K + 64, seed=11)
    At = dev_bf16(A)[:, 16:16 + K]
    Bt = dev_bf16(B)[:, 64:64 + K]
    Cbig = torch.zeros((M, N + 24), dtype=torch.bfloat16, device="cuda")
    C = Cbig[:, :N]
    g.gemm_bf16(At, Bt, C, variant="band")
    ref = oracle.gemm_bf16(np.ascontiguousarray(A[:, 16:16 + K]), np.ascontiguousarray(B[:, 64:64 + K]))
    assert_close(host_bits(C), ref, what=f"band strided {M}x{N}x{K}")
    assert not host_bits(Cbig[:, N:]).any()     # nothing written past N


def test_leading_dimensions_and_views(g):
    import torch
    M, N, K = 37, 200, 96
    A, B = bf16_inputs(M, N + 8, K + 16, seed=3)
    At = dev_bf16(A)[:, 8:8 + K]          # lda = K + 16, 16-byte aligned offset
    Bt = dev_bf16(B)[:N, 16:16 + K]
    Cbig = torch.zeros((M, N + 24), dtype=torch.bfloat16, device="cuda")
    C = Cbig[:, :N]
    g.gemm_bf16(At, Bt, C)
    ref = oracle.gemm_bf16(np.ascontiguousarray(A[:, 8:8 + K]), np.ascontiguousarray(B[:N, 16:16 + K]))
    assert_close(host_bits(C), ref, what="strided")
    assert not host_bits(Cbig[:, N:]).any()     # nothing written past N


# Odd N (C padded to a leading dimension that is a multiple of 8) under cluster
# split-K of 8, 4, 2 and 3 CTAs: the reduction stores neighbouring output columns
# in pairs where the split allows, and the last column of an odd N pairs with none.
ODD_N = [(8, 1001, 4096), (64, 255, 2048), (128, 383, 8192), (8, 4863, 1024), (32, 9727, 512),
         (16, 6399, 768)]


@pytest.mark.parametrize("M,N,K", ODD_N)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_odd_n_split_reduction(g, M, N, K, kind):
    import torch
    A, B = bf16_inputs(M, N, K, seed=M + N, kind=kind)
    ldc = (N + 7) // 8 * 8 + 8
    Cbig = torch.zeros((M, ldc), dtype=torch.bfloat16, device="cuda")
    C = Cbig[:, :N]
    g.gemm_bf16(dev_bf16(A), dev_bf16(B), C, variant="skinny")
    ref = oracle.gemm_bf16(A, B)
    (assert_exact if kind == "int" else assert_close)(host_bits(C), ref, what=f"odd N {M}x{N}x{K}")
    assert not host_bits(Cbig[:, N:]).any()     # nothing written past N


def test_k_zero_and_empty(g):
    import torch
    C = torch.full((5, 24), 3.0, dtype=torch.bfloat16, device="cuda")
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((24, 0), dtype=torch.bfloat16, device="cuda")
    g.gemm_bf16(A, B, C)
    assert not host_bits(C).any()
    E = g.gemm_bf16(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                    torch.empty((24, 64), dtype=torch.bfloat16, device="cuda"))
    assert E.shape == (0, 24)


@pytest.mark.parametrize("variant", VARIANTS)
def test_deterministic(g, variant):
    M, N, K = 96, 4096, 4096
    if not runnable(g, M, N, K, variant):
        pytest.skip("variant does not run")
    A, B = bf16_inputs(M, N, K, seed=11)
    dA, dB = dev_bf16(A), dev_bf16(B)
    c1 = host_bits(g.gemm_bf16(dA, dB, variant=variant))
    c2 = host_bits(g.gemm_bf16(dA, dB, variant=variant))
    assert np.array_equal(c1, c2)


# ------------------------------------------------------------ full-size configs

DECODE = [(M, N, 4096) for M in (1, 8, 32, 128) for N in (6144, 4096, 24576)]
DOWN = [(M, 4096, 12288) for M in (1, 16, 64, 128, 512)]
PREFILL = [(M, N, K) for M in (1024, 4096, 16384)
           for (N, K) in ((4096, 4096), (6144, 4096), (24576, 4096), (4096, 12288), (8192, 8192))]


class Inputs:
    """Largest draw per K, sliced per shape (draws are counter-based, so the
    first rows of a larger draw equal a smaller draw of the same K)."""
    cache = {}

    @classmethod
    def get(cls, M, N, K, kind):
        key = (K, kind)
        if key not in cls.cache:
            Mmax = max(m for (m, _, k) in DECODE + DOWN + PREFILL if k == K)
            Nmax = max(n for (_, n, k) in DECODE + DOWN + PREFILL if k == K)
            A, B = bf16_inputs(Mmax, Nmax, K, seed=0, kind=kind)
            cls.cache = {key: (A, B, dev_bf16(A), dev_bf16(B))}   # keep one K resident
        A, B, dA, dB = cls.cache[key]
        return A[:M], B[:N], dA[:M], dB[:N]


def check_full(g, M, N, K, kind):
    A, B, dA, dB = Inputs.get(M, N, K, kind)
    C = host_bits(g.gemm_bf16(dA, dB))
    ref = oracle.gemm_bf16(A, B)
    (assert_exact if kind == "int" else assert_close)(C, ref, what=f"{M}x{N}x{K}")


def check_sampled(g, M, N, K, kind):
    A, B, dA, dB = Inputs.get(M, N, K, kind)
    C = host_bits(g.gemm_bf16(dA, dB))
    rows = sample_rows(M, 3, seed=M + N)
    cols = sample_rows(N, 3, seed=K)
    ref_r = oracle.gemm_bf16(A[rows], B)
    ref_c = oracle.gemm_bf16(A, B[cols])
    if kind == "int":
        assert_exact(C[rows], ref_r, what=f"rows {M}x{N}x{K}")
        assert_exact(C[:, cols], ref_c, what=f"cols {M}x{N}x{K}")
    else:
        rms = float(np.sqrt(np.mean(np.concatenate([ref_r.ravel(), ref_c.ravel()]) ** 2)))
        assert_close(C[rows], ref_r, rms, what=f"rows {M}x{N}x{K}")
        assert_close(C[:, cols], ref_c, rms, what=f"cols {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", DECODE + DOWN)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_full_size_decode(g, M, N, K, kind):
    check_full(g, M, N, K, kind)


@pytest.mark.parametrize("M,N,K", PREFILL)
@pytest.mark.parametrize("kind", ["normal", "int"])
def test_full_size_prefill(g, M, N, K, kind):
    if not runnable(g, M, N, K, "auto"):
        pytest.skip("no tensor-core plan for this shape yet")
    (check_full if M <= 1024 else check_sampled)(g, M, N, K, kind)


def test_pr1_reference_case(g):
    # 256^3, N(0,1) inputs (seed 0) and integer inputs in [-4,4]
    for kind in ("normal", "int"):
        A, B = bf16_inputs(256, 256, 256, seed=0, kind=kind)
        if kind == "normal":
            from dense_bit_weight_gb300 import synth
            B = synth.bf16_normal((256, 256), 1.0, 0, synth.STREAM_B)   # both N(0,1)
        C = host_bits(g.gemm_bf16(dev_bf16(A), dev_bf16(B)))
        ref = oracle.gemm_bf16(A, B)
        (assert_exact if kind == "int" else assert_close)(C, ref, what=f"PR1 {kind}")
