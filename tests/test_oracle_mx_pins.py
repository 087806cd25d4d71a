"""Pins of the block-scaled (MX) oracle against things other than itself.

FlyDSL-in-PyTorch blog, section "MXFP": FP8 E4M3 or packed FP4 E2M1 operands,
one E8M0 scale per 32 values along K, fp32 accumulation; the element formats
are the OCP microscaling ones.  Pinned here:
  - every E4M3 code against torch's float8_e4m3fn conversion (a library routine)
  - the sixteen E2M1 codes against the OCP value table, written out
  - every E8M0 code against math.ldexp
  - unit scales and integer elements: the int64 matmul, exactly
  - power-of-two scales: the (separately pinned) bf16 oracle on the decoded,
    pre-scaled operands, bit for bit (the same exact products in the same order)
  - one scale moved by 2^1: the result moves by exactly that block's partial sum
    (catches a wrong block index or block length)
  - a single set E2M1 nibble: the low nibble of byte j is element 2j, the high
    one element 2j + 1
  - tiny random cases: exact rational arithmetic (fractions) within the fp64
    summation bound
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from dense_bit_weight_gb300 import synth


def test_e4m3_decode_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.mx_decode(codes, "e4m3")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0


def test_e2m1_decode_matches_ocp_table():
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    codes = np.arange(16, dtype=np.uint8)
    got = oracle.mx_decode(codes, "e2m1")
    assert np.array_equal(got[:8], table)
    assert np.array_equal(got[8:], [-v for v in table])
    assert math.copysign(1.0, got[8]) == -1.0          # code 8 is -0


def test_e8m0_decode_matches_ldexp():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.mx_decode(codes, "e8m0")
    assert math.isnan(got[255])
    assert all(got[e] == math.ldexp(1.0, e - 127) for e in range(255))


def decoded(el, fmt):
    """[rows, K] fp64 element values, decoded code by code through the oracle's
    (pinned) decoder; packed E2M1 unpacked low nibble first."""
    if fmt == "e4m3":
        return oracle.mx_decode(el, "e4m3")
    lo = oracle.mx_decode(el & 0xF, "e2m1")
    hi = oracle.mx_decode(el >> 4, "e2m1")
    out = np.empty((el.shape[0], 2 * el.shape[1]))
    out[:, 0::2], out[:, 1::2] = lo, hi
    return out


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e2m1", "e2m1"), ("e4m3", "e2m1")])
@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 64), (17, 9, 256)])
def test_unit_scales_integers_equal_int64_matmul(fa, fb, M, N, K):
    A, SA = synth.mx_operands(M, K, fa, seed=M + K, role="a", kind="int")
    B, SB = synth.mx_operands(N, K, fb, seed=N + K, role="b", kind="int")
    ia = decoded(A, fa).astype(np.int64)
    ib = decoded(B, fb).astype(np.int64)
    assert np.array_equal(decoded(A, fa), ia) and np.abs(ia).max() <= 4
    want = ia @ ib.T
    got = oracle.gemm_mx(A, SA, B, SB, fa, fb)
    assert np.array_equal(got, want.astype(np.float64))


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e2m1", "e2m1")])
def test_power_of_two_scales_equal_bf16_oracle(fa, fb):
    M, N, K = 7, 11, 320
    A, SA = synth.mx_operands(M, K, fa, seed=3, role="a")
    B, SB = synth.mx_operands(N, K, fb, seed=4, role="b")
    sa = np.repeat(oracle.mx_decode(SA, "e8m0"), 32, axis=1)
    sb = np.repeat(oracle.mx_decode(SB, "e8m0"), 32, axis=1)
    av, bv = decoded(A, fa) * sa, decoded(B, fb) * sb
    # every pre-scaled value is exact in bf16 (at most 4 significant bits, |e| small)
    to_bf16 = lambda x: (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    abits, bbits = to_bf16(av), to_bf16(bv)
    assert np.array_equal(oracle.bf16_bits_to_f64(abits), av)
    assert np.array_equal(oracle.bf16_bits_to_f64(bbits), bv)
    assert np.array_equal(oracle.gemm_mx(A, SA, B, SB, fa, fb), oracle.gemm_bf16(abits, bbits))


def test_one_scale_moves_exactly_its_block():
    M, N, K = 2, 3, 128
    A, SA = synth.mx_operands(M, K, "e4m3", seed=5, role="a", kind="int")
    B, SB = synth.mx_operands(N, K, "e4m3", seed=6, role="b", kind="int")
    base = oracle.gemm_mx(A, SA, B, SB)
    ia, ib = decoded(A, "e4m3").astype(np.int64), decoded(B, "e4m3").astype(np.int64)
    for (m, j) in [(0, 0), (1, 2), (1, 3)]:
        SA2 = SA.copy()
        SA2[m, j] = 128                      # 2^1 instead of 2^0
        moved = oracle.gemm_mx(A, SA2, B, SB) - base
        block = ia[m, 32 * j:32 * j + 32] @ ib[:, 32 * j:32 * j + 32].T
        want = np.zeros_like(base)
        want[m] = block
        assert np.array_equal(moved, want.astype(np.float64))


@pytest.mark.parametrize("k", [0, 1, 30, 31, 62, 63])
def test_e2m1_nibble_order(k):
    N, K = 4, 64
    A = np.zeros((1, K // 2), np.uint8)
    A[0, k // 2] = 0x2 << (4 * (k % 2))      # element k = 1.0
    SA = np.full((1, K // 32), 127, np.uint8)
    B, SB = synth.mx_operands(N, K, "e2m1", seed=7, role="b", kind="int")
    got = oracle.gemm_mx(A, SA, B, SB, "e2m1", "e2m1")
    assert np.array_equal(got[0], decoded(B, "e2m1")[:, k])


@pytest.mark.parametrize("fa,fb", [("e4m3", "e4m3"), ("e2m1", "e4m3")])
def test_random_against_exact_rationals(fa, fb):
    M, N, K = 2, 3, 96
    A, SA = synth.mx_operands(M, K, fa, seed=8, role="a")
    B, SB = synth.mx_operands(N, K, fb, seed=9, role="b")
    av = decoded(A, fa) * np.repeat(oracle.mx_decode(SA, "e8m0"), 32, axis=1)
    bv = decoded(B, fb) * np.repeat(oracle.mx_decode(SB, "e8m0"), 32, axis=1)
    got = oracle.gemm_mx(A, SA, B, SB, fa, fb)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(av[m, k])) * Fraction(float(bv[n, k])) for k in range(K))
            bound = K * 2.0 ** -53 * float(sum(abs(av[m, k] * bv[n, k]) for k in range(K)))
            assert abs(Fraction(float(got[m, n])) - exact) <= Fraction(bound)


def test_rejects_bad_shapes():
    A = np.zeros((2, 48), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_mx(A, np.zeros((2, 1), np.uint8), A, np.zeros((2, 1), np.uint8))
