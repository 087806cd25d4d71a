"""Pins of the fp64 CPU oracle against things other than itself.

Each test fixes the oracle to exact integer arithmetic (numpy int64 matmul),
exact rational arithmetic (fractions.Fraction on tiny inputs), closed forms
(identity operands, a single set nibble), invariants (permutations, linearity,
thread count) or a library routine (numpy float64 matmul, torch's bf16 cast).
A dropped term, a wrong sign or index, a transposed operand or a wrong nibble
or group index in the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from dense_bit_weight_gb300 import synth

F64 = oracle.bf16_bits_to_f64


def ints(shape, stream, lo=-4, hi=4, seed=0):
    v = synth.int_uniform(shape, lo, hi, seed, stream)
    return v, synth.bf16_from_small_ints(v)


# ------------------------------------------------------------- bf16 rounding

def test_round_known_values():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    vals = [1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40, -2.5, 0.0, -0.0,
            2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 3.4e38, 3.5e38, 1e39, -1e39]
    want = [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0x8000,
            0x0001, 0x0000, 0x0002, 0x7F80 if 3.4e38 >= 2 ** 128 * (1 - 2 ** -9) else 0x7F7F,
            0x7F80, 0x7F80, 0xFF80]
    got = oracle.round_to_bf16(np.array(vals))
    assert [int(x) for x in got] == want


def test_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    # values exactly representable in fp32, so torch's fp32 -> bf16 cast is a
    # single RNE rounding, as is the oracle's fp64 -> bf16
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add exact ties: low 16 bits == 0x8000
    ties = ((bits[:5000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    f = np.concatenate([f, ties[np.isfinite(ties)]])
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_single_rounding_from_fp64():
    # x = 1 + 2^-8 + 2^-30 rounds up to 1 + 2^-7 directly, but through fp32 it
    # would first become 1 + 2^-8 (a tie) and then round down to 1.0
    x = 1 + 2 ** -8 + 2 ** -30
    assert int(oracle.round_to_bf16(np.array([x]))[0]) == 0x3F81
    # brute force against exact rationals on random fp64 in a few binades
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(2000) * np.exp2(rng.integers(-20, 20, 2000))
    got = oracle.round_to_bf16(xs)
    for x, g in zip(xs, got):
        fx = Fraction(float(x))
        e = Fraction(abs(fx)).numerator.bit_length() - Fraction(abs(fx)).denominator.bit_length()
        # find the binade exactly
        while Fraction(2) ** e > abs(fx):
            e -= 1
        while Fraction(2) ** (e + 1) <= abs(fx):
            e += 1
        q = Fraction(2) ** (e - 7)
        r = fx / q
        fl = r.numerator // r.denominator
        rem = r - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        exact = float(fl * q)
        assert F64(np.array([g], dtype=np.uint16))[0] == exact


# ------------------------------------------------------------- bf16 GEMM

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 7, 8), (17, 8, 24), (33, 16, 136),
                                   (64, 136, 256), (5, 300, 1000)])
def test_integer_exact_vs_int64_matmul(M, N, K):
    a, A = ints((M, K), 11)
    b, B = ints((N, K), 12)
    R = oracle.gemm_bf16(A, B)
    assert np.array_equal(R, (a @ b.T).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 7), (7, 8, 16), (8, 16, 33), (16, 33, 3)])
def test_brute_force_exact_rationals(M, N, K):
    A = synth.bf16_normal((M, K), 1.0, 3, 1)
    B = synth.bf16_normal((N, K), 0.5, 3, 2)
    R = oracle.gemm_bf16(A, B)
    a, b = F64(A), F64(B)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(float(a[m, k])) * Fraction(float(b[n, k])) for k in range(K)),
                        Fraction(0))
            bound = K * 2.0 ** -53 * float(np.sum(np.abs(a[m] * b[n])))
            assert abs(Fraction(float(R[m, n])) - exact) <= Fraction(bound)


def test_float_vs_numpy_blas():
    M, N, K = 37, 53, 1024
    A = synth.bf16_normal((M, K), 1.0, 5, 1)
    B = synth.bf16_normal((N, K), K ** -0.5, 5, 2)
    R = oracle.gemm_bf16(A, B)
    ref = F64(A) @ F64(B).T
    assert np.max(np.abs(R - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


def test_identity_operands():
    K = 40
    eye = synth.bf16_from_small_ints(np.eye(K, dtype=np.int64))
    B = synth.bf16_normal((23, K), 1.0, 7, 2)
    A = synth.bf16_normal((19, K), 1.0, 7, 1)
    assert np.array_equal(oracle.gemm_bf16(eye, B), F64(B).T)   # A = I  ->  C = B^T
    assert np.array_equal(oracle.gemm_bf16(A, eye), F64(A))     # B = I  ->  C = A


def test_permutation_invariants():
    M, N, K = 13, 29, 96
    rng = np.random.default_rng(2)
    A = synth.bf16_normal((M, K), 1.0, 9, 1)
    B = synth.bf16_normal((N, K), 1.0, 9, 2)
    R = oracle.gemm_bf16(A, B)
    pm, pn, pk = rng.permutation(M), rng.permutation(N), rng.permutation(K)
    assert np.array_equal(oracle.gemm_bf16(A[pm], B), R[pm])
    assert np.array_equal(oracle.gemm_bf16(A, B[pn]), R[:, pn])
    Rk = oracle.gemm_bf16(A[:, pk], B[:, pk])
    assert np.max(np.abs(Rk - R)) <= 1e-12 * np.sqrt(np.mean(R ** 2))
    a, Ai = ints((M, K), 11)
    b, Bi = ints((N, K), 12)
    assert np.array_equal(oracle.gemm_bf16(Ai[:, pk], Bi[:, pk]), oracle.gemm_bf16(Ai, Bi))


def test_linearity_on_integers():
    M, N, K = 9, 31, 64
    a1, _ = ints((M, K), 21, -2, 2)
    a2, _ = ints((M, K), 22, -2, 2)
    b, B = ints((N, K), 23)
    cat = lambda v: synth.bf16_from_small_ints(v)
    lhs = oracle.gemm_bf16(cat(a1 + a2), B)
    rhs = oracle.gemm_bf16(cat(a1), B) + oracle.gemm_bf16(cat(a2), B)
    assert np.array_equal(lhs, rhs)


def test_gemv_and_outer_product_special_cases():
    K = 777
    A = synth.bf16_normal((1, K), 1.0, 11, 1)
    B = synth.bf16_normal((50, K), 1.0, 11, 2)
    R = oracle.gemm_bf16(A, B)
    ref = F64(B) @ F64(A)[0]                       # textbook GEMV
    assert np.max(np.abs(R[0] - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))
    A1 = synth.bf16_normal((6, 1), 1.0, 12, 1)
    B1 = synth.bf16_normal((9, 1), 1.0, 12, 2)
    assert np.array_equal(oracle.gemm_bf16(A1, B1), np.outer(F64(A1)[:, 0], F64(B1)[:, 0]))


def test_empty_and_thread_invariance():
    A = synth.bf16_normal((0, 16), 1.0, 1, 1)
    B = synth.bf16_normal((5, 16), 1.0, 1, 2)
    assert oracle.gemm_bf16(A, B).shape == (0, 5)
    Z = oracle.gemm_bf16(np.zeros((3, 0), np.uint16), np.zeros((4, 0), np.uint16))
    assert np.array_equal(Z, np.zeros((3, 4)))     # K = 0: the empty sum
    A = synth.bf16_normal((41, 200), 1.0, 2, 1)
    B = synth.bf16_normal((37, 200), 1.0, 2, 2)
    assert np.array_equal(oracle.gemm_bf16(A, B, threads=1), oracle.gemm_bf16(A, B, threads=7))


# ------------------------------------------------------------- W4A16

def _pack(q):
    """Pack a [N,K] array of nibbles per the stated layout (test-side packer)."""
    N, K = q.shape
    w = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        w |= (q[:, j::8].astype(np.uint32) & np.uint32(15)) << np.uint32(4 * j)
    return w.view(np.int32)


def test_w4_single_nibble_fixes_layout():
    # one nibble set at word w, position j must pick up A[:, 8w + j]
    M, N, K, g = 3, 2, 64, 32
    A = synth.bf16_normal((M, K), 1.0, 4, 1)
    a = F64(A)
    one = synth.bf16_from_small_ints(np.ones((N, K // g), np.int64))
    for w, j in [(0, 0), (0, 7), (3, 1), (7, 4)]:
        Bq = np.zeros((N, K // 8), dtype=np.uint32)
        Bq[1, w] = np.uint32(5) << np.uint32(4 * j)
        R = oracle.gemm_w4a16(A, Bq.view(np.int32), one, np.zeros((N, K // g), np.uint8), g)
        assert np.array_equal(R[:, 0], np.zeros(M))
        assert np.array_equal(R[:, 1], 5.0 * a[:, 8 * w + j])


def test_w4_group_index_and_zero_sign():
    # q = 0 everywhere, z = 1 in group 1 only, s = 2^t per group:
    # w[n,k] = -(z) * s = -2 on group 1, 0 elsewhere
    M, N, K, g = 2, 3, 128, 32
    A = synth.bf16_normal((M, K), 1.0, 6, 1)
    a = F64(A)
    Bq = np.zeros((N, K // 8), dtype=np.int32)
    zeros = np.zeros((N, K // g), np.uint8)
    zeros[:, 1] = 1
    scales = synth.bf16_from_small_ints(np.array([[1, 2, 4, 8]] * N))
    R = oracle.gemm_w4a16(A, Bq, scales, zeros, g)
    want = -2.0 * a[:, g:2 * g].sum(axis=1)
    for n in range(N):
        assert np.allclose(R[:, n], want, rtol=0, atol=1e-12)


def test_w4_unit_scale_zero8_equals_bf16_oracle():
    M, N, K, g = 7, 45, 256, 128
    q = synth.int_uniform((N, K), 0, 15, 0, 31)
    a, A = ints((M, K), 32)
    Bq = _pack(q)
    one = synth.bf16_from_small_ints(np.ones((N, K // g), np.int64))
    z8 = np.full((N, K // g), 8, np.uint8)
    R = oracle.gemm_w4a16(A, Bq, one, z8, g)
    assert np.array_equal(R, oracle.gemm_bf16(A, synth.bf16_from_small_ints(q - 8)))
    assert np.array_equal(R, (a @ (q - 8).T).astype(np.float64))


@pytest.mark.parametrize("g", [32, 64, 128])
def test_w4_integer_exact_with_power_of_two_scale(g):
    M, N, K = 4, 33, 512
    a, A = ints((M, K), 41)
    Bq, _, zeros = synth.w4a16_operands(N, K, g, seed=3)
    s = synth.bf16_from_small_ints(np.ones((N, K // g), np.int64))
    s = (s.astype(np.uint32) - np.uint32(4 << 7)).astype(np.uint16)   # 1.0 * 2^-4 exactly
    assert F64(s)[0, 0] == 2.0 ** -4
    q = ((Bq.view(np.uint32)[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15)
    q = q.reshape(N, K).astype(np.int64)
    zk = np.repeat(zeros.astype(np.int64), g, axis=1)
    want = (a @ (q - zk).T).astype(np.float64) * 2.0 ** -4
    assert np.array_equal(oracle.gemm_w4a16(A, Bq, s, zeros, g), want)


def test_w4_general_vs_dequant_and_blas():
    M, N, K, g = 5, 70, 1024, 128
    A = synth.bf16_normal((M, K), 1.0, 8, 1)
    Bq, s, z = synth.w4a16_operands(N, K, g, seed=8)
    R = oracle.gemm_w4a16(A, Bq, s, z, g)
    W = oracle.dequant_w4(Bq, s, z, g)
    # dequantised weights against a vectorised decode of the stated layout
    q = ((Bq.view(np.uint32)[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 15)
    q = q.reshape(N, K).astype(np.float64)
    Wv = (q - np.repeat(z.astype(np.float64), g, 1)) * np.repeat(F64(s), g, 1)
    assert np.array_equal(W, Wv)
    ref = F64(A) @ W.T
    assert np.max(np.abs(R - ref)) <= 1e-12 * np.sqrt(np.mean(ref ** 2))


# ------------------------------------------------------------- tolerance helper

# ------------------------------------------------------ fused epilogues

def test_silu_textbook_values():
    # silu(x) = x * sigmoid(x); sigmoid(1) = 1 / (1 + 1/e) = 0.7310585786300049
    g = np.array([0.0, 1.0, -1.0, 2.0])
    got = oracle.silu_mul(g, np.array([1.0, 1.0, 1.0, 0.5]))
    want = [0.0, 0.7310585786300049, -0.2689414213699951, 0.5 * 2.0 * 0.8807970779778823]
    assert np.allclose(got, want, rtol=1e-15, atol=0)


def test_silu_tanh_form_and_odd_part():
    # two closed forms independent of the oracle's: silu(x) = (x/2)(1 + tanh(x/2)),
    # and silu(x) - silu(-x) = x (a sign or exponent error breaks both)
    # (the tanh form cancels for large negative x; there x e^x / (1 + e^x) is exact-ish)
    x = np.linspace(-30.0, 30.0, 1201)
    one = np.ones_like(x)
    s = oracle.silu_mul(x, one)
    pos = x >= -4.0
    assert np.allclose(s[pos], 0.5 * x[pos] * (1.0 + np.tanh(0.5 * x[pos])), rtol=1e-13, atol=1e-300)
    neg = x < 0.0
    ex = np.exp(x[neg])
    assert np.allclose(s[neg], x[neg] * ex / (1.0 + ex), rtol=1e-13, atol=1e-300)
    assert np.allclose(s - oracle.silu_mul(-x, one), x, rtol=1e-14, atol=1e-14)
    # saturation: silu(-1000) is -0 (not NaN), silu(1000) = 1000
    assert np.array_equal(oracle.silu_mul(np.array([-1000.0, 1000.0]), np.ones(2)), [-0.0, 1000.0])


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (5, 24, 40), (33, 136, 264)])
def test_bias_epilogue_integer_exact(M, N, K):
    a, A = ints((M, K), 11)
    b, B = ints((N, K), 12)
    c, Cb = ints((N,), 13, -40, 40)
    R = oracle.gemm_bf16_bias(A, B, Cb)
    assert np.array_equal(R, (a @ b.T + c[None, :]).astype(np.float64))


def test_bias_epilogue_vs_blas():
    A = synth.bf16_normal((17, 96), 1.0, 4, 1)
    B = synth.bf16_normal((40, 96), 0.1, 4, 2)
    bias = synth.bf16_normal((40,), 1.0, 4, 3)
    want = F64(A) @ F64(B).T + F64(bias)[None, :]
    assert np.allclose(oracle.gemm_bf16_bias(A, B, bias), want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (7, 24, 40), (16, 72, 128)])
def test_silu_mul_gate_up_layout(M, N, K):
    # B stacks the gate rows (0..N-1) over the up rows (N..2N-1): g and u are
    # exact integer sums here, and the tanh form is independent of the oracle
    a, A = ints((M, K), 21)
    b, B = ints((2 * N, K), 22)
    g = (a @ b[:N].T).astype(np.float64)
    u = (a @ b[N:].T).astype(np.float64)
    want = 0.5 * g * (1.0 + np.tanh(0.5 * g)) * u
    got = oracle.gemm_bf16_silu_mul(A, B)
    assert got.shape == (M, N)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-12)
    # the halves are not interchangeable (the test would catch a swapped layout)
    swapped = 0.5 * u * (1.0 + np.tanh(0.5 * u)) * g
    assert not np.allclose(got, swapped, rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------ grouped GEMM

@pytest.mark.parametrize("sizes", [[5, 0, 17, 3], [0, 0, 9], [32], [1, 1, 1, 1, 1, 1, 1, 1]])
def test_grouped_integer_exact_per_expert(sizes):
    # every row against an int64 matmul with its own expert's weights; rows
    # past the last expert stay 0
    G, N, K = len(sizes), 24, 40
    ends = np.cumsum(sizes).astype(np.int32)
    M = int(ends[-1]) + 3
    a, A = ints((M, K), 31)
    b, B = ints((G, N, K), 32)
    R = oracle.gemm_grouped(A, B, ends)
    want = np.zeros((M, N))
    start = 0
    for g, e in enumerate(ends):
        want[start:e] = a[start:e] @ b[g].T
        start = e
    assert np.array_equal(R, want)


def test_grouped_one_expert_is_the_plain_gemm_and_order_matters():
    a, A = ints((20, 32), 33)
    b, B = ints((2, 16, 32), 34)
    assert np.array_equal(oracle.gemm_grouped(A, B[:1], np.array([20], np.int32)), oracle.gemm_bf16(A, B[0]))
    # moving the boundary moves rows between experts (an off-by-one in the
    # row ranges fails this)
    r1 = oracle.gemm_grouped(A, B, np.array([7, 20], np.int32))
    r2 = oracle.gemm_grouped(A, B, np.array([8, 20], np.int32))
    assert np.array_equal(r1[:7], r2[:7]) and np.array_equal(r1[8:], r2[8:])
    assert np.array_equal(r1[7], (a[7] @ b[1].T).astype(np.float64))
    assert np.array_equal(r2[7], (a[7] @ b[0].T).astype(np.float64))


def test_grouped_rejects_bad_offsets():
    _, A = ints((4, 8), 35)
    _, B = ints((2, 8, 8), 36)
    for bad in ([3, 2], [2, 5], [-1, 4]):
        with pytest.raises(RuntimeError):
            oracle.gemm_grouped(A, B, np.array(bad, np.int32))


# ------------------------------------------------------------ bias + activation epilogues

def test_bias_relu_integer_exact():
    M, N, K = 5, 33, 64
    A = synth.bf16_int_uniform((M, K), -4, 4, 1, synth.STREAM_A_INT)
    B = synth.bf16_int_uniform((N, K), -4, 4, 1, synth.STREAM_B_INT)
    bias = synth.bf16_int_uniform((N,), -40, 40, 2, synth.STREAM_B_INT)
    ia = oracle.bf16_bits_to_f64(A).astype(np.int64)
    ib = oracle.bf16_bits_to_f64(B).astype(np.int64)
    pre = ia @ ib.T + oracle.bf16_bits_to_f64(bias).astype(np.int64)
    got = oracle.gemm_bf16_bias_act(A, B, bias, "relu")
    assert np.array_equal(got, np.maximum(pre, 0).astype(np.float64))
    assert (got == 0).any() and (got > 0).any()


def test_bias_silu_tanh_form():
    x = np.linspace(-30.0, 30.0, 601).reshape(1, -1)
    bias = synth.bf16_from_small_ints(np.arange(601) % 7 - 3)
    xb = x + oracle.bf16_bits_to_f64(bias)
    got = oracle.bias_act(x, bias, "silu")
    assert np.allclose(got, xb / 2 * (1 + np.tanh(xb / 2)), rtol=1e-12, atol=1e-12)
    neg = xb < 0   # the stable form for negative x, exact relative agreement
    assert np.allclose(got[neg], (xb * np.exp(xb) / (1 + np.exp(xb)))[neg], rtol=1e-13, atol=0)


def test_bias_gelu_against_library_and_invariants():
    x = np.linspace(-12.0, 12.0, 481).reshape(1, -1)
    zero = np.zeros(x.shape[1], np.uint16)
    got = oracle.bias_act(x, zero, "gelu")
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="none").numpy()
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-15)
    # x Phi(x) - (-x) Phi(-x) = x, and the textbook value at 1
    neg = oracle.bias_act(-x, zero, "gelu")
    assert np.allclose(got - neg, x, rtol=1e-13, atol=1e-13)
    one = oracle.bias_act(np.array([[1.0]]), np.zeros(1, np.uint16), "gelu")
    assert abs(one[0, 0] - 0.8413447460685429) < 1e-15
    # the bias is added before the activation
    b = synth.bf16_from_small_ints(np.full(x.shape[1], 2))
    assert np.allclose(oracle.bias_act(x, b, "gelu"), oracle.bias_act(x + 2.0, zero, "gelu"), rtol=1e-15, atol=0)


def test_tolerance_flags_planted_error():
    ref = synth.normal_f64(1000, 0, 9).reshape(10, 100)
    out = ref.copy()
    ok, rms = oracle.within_tolerance(out, ref)
    assert ok.all()
    out[3, 7] = ref[3, 7] + 0.03 * abs(ref[3, 7]) + 0.011 * rms
    ok, _ = oracle.within_tolerance(out, ref)
    assert not ok[3, 7] and ok.sum() == ok.size - 1
