"""GPU parity of gemm_bf16_fused (bias and SiLU-mul epilogues) against the fp64 oracle.

Small and ragged shapes are compared element by element for every kernel
family and split path (GEMV; skinny tcgen05 with whole tiles, cluster split-K
and stream-K; prefill tcgen05 with whole tiles and stream-K; CTA pairs with
whole tiles and stream-K).  The decode and
prefill gate/up projections run at full size: every element of C up to
M = 1024, sampled rows and columns at M = 4096.  Integer-valued inputs with a bias are exact; everything else
must satisfy |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).
"""
import numpy as np
import pytest

import oracle
from dense_bit_weight_gb300 import synth
from gpu_helpers import assert_close, assert_exact, bf16_inputs, dev_bf16, host_bits, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import torch
    from dense_bit_weight_gb300 import gemm
    torch.cuda.init()
    yield gemm
    assert gemm.gemm_last_device_error() == 0


def plan_of(g, M, NB, K, variant):
    try:
        return g.gemm_bf16_plan(M, NB, K, variant)
    except g.GemmError:
        return None


# (M, N, K): N = columns of C; the SiLU-mul weight has 2N rows
SMALL = [(1, 8, 16), (3, 72, 264), (4, 1000, 136),               # GEMV
         (8, 40, 512), (16, 520, 1032), (33, 4104, 72),          # skinny, whole tiles / cluster split
         (128, 200, 4096), (8, 20480, 512),                      # skinny, split 8 / stream-K (320 tiles)
         (129, 264, 72), (300, 1200, 4096), (1000, 136, 136),    # prefill, stream-K
         (2048, 2048, 1024)]                                     # prefill, whole tiles
VARIANTS = ["gemv", "skinny", "prefill", "pair", "band"]


def runnable(g, M, NB, K, variant):
    p = plan_of(g, M, NB, K, variant)
    return p is not None and not (p["variant"] == 1 and M > 64)


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("kind", ["int", "normal"])
def test_bias(g, M, N, K, variant, kind):
    if not runnable(g, M, N, K, variant):
        pytest.skip(f"{variant} does not run {M}x{N}x{K}")
    A, B = bf16_inputs(M, N, K, seed=M + 3 * N + K, kind=kind)
    if kind == "int":
        bias = synth.bf16_int_uniform((N,), -40, 40, 5, synth.STREAM_B_INT)
    else:
        bias = synth.bf16_normal((N,), 1.0, 5, synth.STREAM_B)
    C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), dev_bf16(bias), epilogue="bias", variant=variant)
    ref = oracle.gemm_bf16_bias(A, B, bias)
    (assert_exact if kind == "int" else assert_close)(host_bits(C), ref, what=f"bias {variant} {M}x{N}x{K}")


# bias + activation (the guide's bias_relu, bias_silu, bias_gelu) on every
# store path: GEMV, skinny whole tiles / cluster split-K / stream-K, prefill
# stream-K and whole tiles, and K = 0
ACT_SHAPES = [(3, 72, 264), (16, 520, 1032), (128, 200, 4096), (8, 20480, 512), (300, 1200, 4096),
              (2048, 2048, 1024)]


@pytest.mark.parametrize("M,N,K", ACT_SHAPES)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("act", ["relu", "silu", "gelu"])
def test_bias_activation(g, M, N, K, variant, act):
    if not runnable(g, M, N, K, variant):
        pytest.skip(f"{variant} does not run {M}x{N}x{K}")
    kind = "int" if act == "relu" else "normal"
    A, B = bf16_inputs(M, N, K, seed=M + 5 * N + K, kind=kind)
    if kind == "int":
        bias = synth.bf16_int_uniform((N,), -40, 40, 6, synth.STREAM_B_INT)
    else:
        bias = synth.bf16_normal((N,), 1.0, 6, synth.STREAM_B)
    C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), dev_bf16(bias), epilogue="bias_" + act, variant=variant)
    ref = oracle.gemm_bf16_bias_act(A, B, bias, act)
    (assert_exact if kind == "int" else assert_close)(host_bits(C), ref, what=f"bias_{act} {variant} {M}x{N}x{K}")


@pytest.mark.parametrize("act", ["relu", "silu", "gelu"])
def test_bias_activation_k_zero(g, act):
    import torch
    bias = synth.bf16_normal((24,), 1.0, 2, synth.STREAM_B)
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    C = g.gemm_bf16_fused(A, torch.empty((24, 0), dtype=torch.bfloat16, device="cuda"), dev_bf16(bias),
                          epilogue="bias_" + act)
    ref = oracle.bias_act(np.zeros((5, 24)), bias, act)
    assert_close(host_bits(C), ref, what=f"bias_{act} K=0")


@pytest.mark.parametrize("M,N,K", SMALL)
@pytest.mark.parametrize("variant", VARIANTS)
def test_silu_mul(g, M, N, K, variant):
    try:
        p = g.gemm_bf16_fused_plan(M, N, K, "silu_mul", variant)
    except g.GemmError:
        p = None
    if p is None or (p["variant"] == 1 and M > 64):
        pytest.skip(f"{variant} does not run the SiLU-mul pairs {M}x{2 * N}x{K}")
    A, B = bf16_inputs(M, 2 * N, K, seed=7 * M + N + K)
    C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), epilogue="silu_mul", variant=variant)
    assert tuple(C.shape) == (M, N)
    assert_close(host_bits(C), oracle.gemm_bf16_silu_mul(A, B), what=f"silu_mul {variant} {M}x{N}x{K}")


@pytest.mark.parametrize("variant,M", [("skinny", 16), ("skinny", 64), ("prefill", 512), ("pair", 512)])
def test_silu_mul_splits_keep_pairs(g, variant, M):
    # shapes whose plan splits K: the gate and up rows of a column must be reduced together
    N, K = 64, 8192
    p = g.gemm_bf16_plan(M, 2 * N, K, variant)
    A, B = bf16_inputs(M, 2 * N, K, seed=M)
    C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), epilogue="silu_mul", variant=variant)
    assert_close(host_bits(C), oracle.gemm_bf16_silu_mul(A, B), what=f"split {variant} {p}")


@pytest.mark.parametrize("epilogue", ["bias", "silu_mul"])
def test_wide_single_token_tile(g, epilogue):
    # one token tile: the planner takes 176-row weight tiles (88 gate/up pairs,
    # from 64 tokens on)
    M, N, K = (64, 12280, 64) if epilogue == "silu_mul" else (48, 24560, 64)
    NB = 2 * N if epilogue == "silu_mul" else N
    p = g.gemm_bf16_plan(M, NB, K)
    if p["tile_n"] != 176:
        pytest.skip(f"plan on this device: {p}")
    A, B = bf16_inputs(M, NB, K, seed=5)
    if epilogue == "bias":
        bias = synth.bf16_normal((N,), 1.0, 5, synth.STREAM_B)
        C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), dev_bf16(bias), epilogue="bias")
        ref = oracle.gemm_bf16_bias(A, B, bias)
    else:
        C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), epilogue="silu_mul")
        ref = oracle.gemm_bf16_silu_mul(A, B)
    assert_close(host_bits(C), ref, what=f"wide {epilogue}")


@pytest.mark.parametrize("variant", ["prefill", "pair"])
def test_bias_two_byte_aligned(g, variant):
    # a bias view starting 2 bytes past a 16-byte boundary (the header asks
    # only for 2-byte alignment): the kernels fall back to element loads
    M, N, K = 512, 1024, 256
    A, B = bf16_inputs(M, N, K, seed=13)
    big = synth.bf16_normal((N + 8,), 1.0, 13, synth.STREAM_B)
    dbias = dev_bf16(big)[1:1 + N]
    C = g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), dbias, epilogue="bias_relu", variant=variant)
    ref = oracle.gemm_bf16_bias_act(A, B, big[1:1 + N], "relu")
    assert_close(host_bits(C), ref, what=f"unaligned bias {variant}")


def test_strided_operands_and_padding(g):
    import torch
    M, N, K = 40, 264, 512
    A, B = bf16_inputs(M, 2 * N, K + 16, seed=9)
    At = dev_bf16(A)[:, 8:8 + K]
    Bt = dev_bf16(B)[:, 16:16 + K]
    Cbig = torch.zeros((M, N + 24), dtype=torch.bfloat16, device="cuda")
    g.gemm_bf16_fused(At, Bt, C=Cbig[:, :N], epilogue="silu_mul")
    ref = oracle.gemm_bf16_silu_mul(np.ascontiguousarray(A[:, 8:8 + K]), np.ascontiguousarray(B[:, 16:16 + K]))
    assert_close(host_bits(Cbig[:, :N]), ref, what="strided silu_mul")
    assert not host_bits(Cbig[:, N:]).any()   # nothing written past N


def test_k_zero(g):
    import torch
    bias = synth.bf16_int_uniform((24,), -9, 9, 1, synth.STREAM_B_INT)
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    C = g.gemm_bf16_fused(A, torch.empty((24, 0), dtype=torch.bfloat16, device="cuda"), dev_bf16(bias),
                          epilogue="bias")
    assert np.array_equal(host_bits(C), np.broadcast_to(bias, (5, 24)))
    C = torch.full((5, 24), 3.0, dtype=torch.bfloat16, device="cuda")
    g.gemm_bf16_fused(A, torch.empty((48, 0), dtype=torch.bfloat16, device="cuda"), C=C, epilogue="silu_mul")
    assert not host_bits(C).any()


def test_deterministic(g):
    M, N, K = 96, 2048, 4096
    A, B = bf16_inputs(M, 2 * N, K, seed=2)
    dA, dB = dev_bf16(A), dev_bf16(B)
    c1 = host_bits(g.gemm_bf16_fused(dA, dB, epilogue="silu_mul"))
    c2 = host_bits(g.gemm_bf16_fused(dA, dB, epilogue="silu_mul"))
    assert np.array_equal(c1, c2)


# ------------------------------------------------ full-size gate/up projections

GATE_UP = [(M, 12288, 4096) for M in (1, 8, 32, 128)] + [(1024, 12288, 4096), (4096, 12288, 4096)]


@pytest.mark.parametrize("M,N,K", GATE_UP)
def test_full_size_gate_up(g, M, N, K):
    # decode and M = 1024: every element; M = 4096 (0.8 TMAC): sampled
    A, B = bf16_inputs(M, 2 * N, K, seed=0)
    C = host_bits(g.gemm_bf16_fused(dev_bf16(A), dev_bf16(B), epilogue="silu_mul"))
    if M <= 1024:
        assert_close(C, oracle.gemm_bf16_silu_mul(A, B), what=f"gate/up {M}x{N}x{K}")
        return
    rows = sample_rows(M, 3, seed=M + N)
    cols = sample_rows(N, 3, seed=K)
    ref_r = oracle.gemm_bf16_silu_mul(A[rows], B)
    ref_c = oracle.gemm_bf16_silu_mul(A, np.concatenate([B[cols], B[N + np.asarray(cols)]]))
    rms = float(np.sqrt(np.mean(np.concatenate([ref_r.ravel(), ref_c.ravel()]) ** 2)))
    assert_close(C[rows], ref_r, rms, what=f"gate/up rows {M}x{N}x{K}")
    assert_close(C[:, cols], ref_c, rms, what=f"gate/up cols {M}x{N}x{K}")
