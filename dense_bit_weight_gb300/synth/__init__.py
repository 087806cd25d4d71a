"""Seeded synthetic inputs for the projection GEMM.

This module only draws random numbers and encodes them in the operand formats
the library accepts (bf16 bits, packed 4-bit words, uint8 zero points, bf16
scales).  It holds none of the GEMM's arithmetic; the CUDA path's tests and the
CPU oracle both take their inputs from here.  The generator itself (splitmix64
used counter-style, Box-Muller normals, bf16 rounding through fp32) is
``synth_gen.c``, whose header gives its exact definition.

Because draws are counter-based and row-major, the first M rows of an [M', K]
tensor (M <= M', same K, same stream) equal the [M, K] tensor.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libdbw_synth.so")
_lock = threading.Lock()
_lib = None

# stream ids: one per operand so operands are independent
STREAM_A, STREAM_B, STREAM_Q, STREAM_Z, STREAM_S = 1, 2, 3, 4, 5
STREAM_A_INT, STREAM_B_INT = 11, 12
STREAM_MX_A, STREAM_MX_B, STREAM_MX_SA, STREAM_MX_SB = 21, 22, 23, 24


def build(force: bool = False) -> str:
    """Compile synth_gen.c (gcc, no fast-math) into synth/_build/."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, p, d, i64 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int64
            lib.synth_bf16_normal.argtypes = [u64, u64, u64, u64, d, p]
            lib.synth_bf16_uniform.argtypes = [u64, u64, u64, u64, d, d, p]
            lib.synth_int_uniform.argtypes = [u64, u64, u64, u64, i64, i64, p]
            lib.synth_u32.argtypes = [u64, u64, u64, u64, p]
            lib.synth_normal_f64.argtypes = [u64, u64, u64, u64, p]
            for f in (lib.synth_bf16_normal, lib.synth_bf16_uniform, lib.synth_int_uniform,
                      lib.synth_u32, lib.synth_normal_f64):
                f.restype = None
            _lib = lib
    return _lib


def _n(shape) -> int:
    return int(np.prod(shape, dtype=np.int64))


def normal_f64(count: int, seed: int = 0, stream: int = STREAM_A, start: int = 0) -> np.ndarray:
    """Standard normals number start .. start+count-1 of sequence (seed, stream)."""
    out = np.empty(count, dtype=np.float64)
    _load().synth_normal_f64(seed, stream, start, count, out.ctypes.data)
    return out


def bf16_normal(shape, std: float = 1.0, seed: int = 0, stream: int = STREAM_A) -> np.ndarray:
    """N(0, std^2) rounded to bf16; uint16 bits of the given shape."""
    out = np.empty(_n(shape), dtype=np.uint16)
    _load().synth_bf16_normal(seed, stream, 0, out.size, float(std), out.ctypes.data)
    return out.reshape(shape)


def int_uniform(shape, lo: int, hi: int, seed: int = 0, stream: int = STREAM_A_INT) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive), int64."""
    out = np.empty(_n(shape), dtype=np.int64)
    _load().synth_int_uniform(seed, stream, 0, out.size, int(lo), int(hi), out.ctypes.data)
    return out.reshape(shape)


def bf16_from_small_ints(v) -> np.ndarray:
    """Exact bf16 bits of small integers (|v| <= 256 is exact in bf16)."""
    v = np.asarray(v, dtype=np.int64)
    if v.size and np.abs(v).max() > 256:
        raise ValueError("values not exactly representable in bf16")
    return (v.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_int_uniform(shape, lo: int = -4, hi: int = 4, seed: int = 0,
                     stream: int = STREAM_A_INT) -> np.ndarray:
    """bf16 bits of integers uniform in [lo, hi] (exact)."""
    return bf16_from_small_ints(int_uniform(shape, lo, hi, seed, stream))


def bf16_uniform(shape, lo: float, hi: float, seed: int = 0, stream: int = STREAM_S) -> np.ndarray:
    """U(lo, hi) rounded to bf16 bits."""
    out = np.empty(_n(shape), dtype=np.uint16)
    _load().synth_bf16_uniform(seed, stream, 0, out.size, float(lo), float(hi), out.ctypes.data)
    return out.reshape(shape)


def packed_int4(n_rows: int, k: int, seed: int = 0, stream: int = STREAM_Q) -> np.ndarray:
    """Random packed 4-bit weights, int32 [n_rows, k/8]: every nibble uniform in
    [0, 15] (a uniform 32-bit word holds 8 independent uniform nibbles)."""
    if k % 8:
        raise ValueError("k must be a multiple of 8")
    out = np.empty(n_rows * (k // 8), dtype=np.uint32)
    _load().synth_u32(seed, stream, 0, out.size, out.ctypes.data)
    return out.view(np.int32).reshape(n_rows, k // 8)


def zeros_uint4(n_rows: int, groups: int, seed: int = 0, stream: int = STREAM_Z) -> np.ndarray:
    """Zero points uniform in [0, 15], one per byte: uint8 [n_rows, groups]."""
    return int_uniform((n_rows, groups), 0, 15, seed, stream).astype(np.uint8)


def w4a16_operands(n_rows: int, k: int, group: int = 128, seed: int = 0,
                   scale_lo: float = 0.002, scale_hi: float = 0.02):
    """(Bq, scales_bits, zeros) of the W4A16 workload: q, z uniform in [0,15],
    s ~ U(scale_lo, scale_hi) rounded to bf16."""
    g = k // group
    return (packed_int4(n_rows, k, seed, STREAM_Q),
            bf16_uniform((n_rows, g), scale_lo, scale_hi, seed, STREAM_S),
            zeros_uint4(n_rows, g, seed, STREAM_Z))


# ------------------------------------------------------------ MX (microscaling) operands
# Codes are drawn field by field (sign, exponent, mantissa), so no value is
# computed here; the formats are the OCP ones (E4M3 "fn": s eeee mmm, bias 7;
# E2M1: s ee m, bias 1; E8M0: a biased exponent).

# E4M3 / E2M1 codes of the integers 0..4 (for exactly representable cases)
_E4M3_INT = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48}
_E2M1_INT = {0: 0x0, 1: 0x2, 2: 0x4, 3: 0x5, 4: 0x6}


def e4m3_codes(shape, seed: int = 0, stream: int = STREAM_MX_A, exp_lo: int = 4, exp_hi: int = 10) -> np.ndarray:
    """E4M3 codes with a uniform sign, an exponent field uniform in
    [exp_lo, exp_hi] (the default spans 2^-3 .. 2^3 x 1.m) and a uniform
    3-bit mantissa; exp_hi <= 14 never draws the NaN code.  uint8 of shape."""
    if not 0 <= exp_lo <= exp_hi <= 14:
        raise ValueError("exponent field range must lie in [0, 14]")
    n = _n(shape)
    sgn = int_uniform((n,), 0, 1, seed, stream)
    ex = int_uniform((n,), exp_lo, exp_hi, seed, stream + 100)
    man = int_uniform((n,), 0, 7, seed, stream + 200)
    return ((sgn << 7) | (ex << 3) | man).astype(np.uint8).reshape(shape)


def e2m1_packed(rows: int, k: int, seed: int = 0, stream: int = STREAM_MX_B) -> np.ndarray:
    """Packed E2M1 operand [rows, k/2]: every nibble a uniform 4-bit code
    (all sixteen codes are finite values)."""
    if k % 8:
        raise ValueError("k must be a multiple of 8")
    out = np.empty(rows * (k // 8), dtype=np.uint32)
    _load().synth_u32(seed, stream, 0, out.size, out.ctypes.data)
    return out.view(np.uint8).reshape(rows, k // 2)


def e8m0_codes(shape, lo: int = 124, hi: int = 130, seed: int = 0, stream: int = STREAM_MX_SA) -> np.ndarray:
    """E8M0 scale codes uniform in [lo, hi] (default 2^-3 .. 2^3), uint8."""
    if not 0 <= lo <= hi <= 254:
        raise ValueError("scale codes must lie in [0, 254]")
    return int_uniform(shape, lo, hi, seed, stream).astype(np.uint8)


def mx_int_operand(rows: int, k: int, fmt: str, lo: int = -4, hi: int = 4, seed: int = 0,
                   stream: int = STREAM_MX_A) -> np.ndarray:
    """Integers uniform in [lo, hi] (|v| <= 4) as MX element codes: E4M3 bytes
    [rows, k], or packed E2M1 [rows, k/2] (element k in the low nibble for
    even k)."""
    if not -4 <= lo <= hi <= 4:
        raise ValueError("|v| <= 4")
    v = int_uniform((rows, k), lo, hi, seed, stream)
    table = _E4M3_INT if fmt == "e4m3" else _E2M1_INT
    sign = 0x80 if fmt == "e4m3" else 0x8
    mag = np.vectorize(table.get, otypes=[np.int64])(np.abs(v))
    codes = (mag | np.where(v < 0, sign, 0)).astype(np.uint8)
    if fmt == "e4m3":
        return codes
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def mx_operands(rows: int, k: int, fmt: str, seed: int = 0, role: str = "a", kind: str = "random"):
    """(elements, scales) of one MX operand: random codes with scales in
    2^-3 .. 2^3, or (kind "int") integers in [-4, 4] with unit scales (code
    127), so every product and partial sum is exact."""
    es = STREAM_MX_A if role == "a" else STREAM_MX_B
    ss = STREAM_MX_SA if role == "a" else STREAM_MX_SB
    if kind == "int":
        return mx_int_operand(rows, k, fmt, seed=seed, stream=es), np.full((rows, k // 32), 127, np.uint8)
    el = e4m3_codes((rows, k), seed, es) if fmt == "e4m3" else e2m1_packed(rows, k, seed, es)
    return el, e8m0_codes((rows, k // 32), seed=seed, stream=ss)
