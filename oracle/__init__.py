"""fp64 CPU oracle for the projection GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never links or calls it,
and it shares no code with the CUDA path.

The arithmetic lives in ``oracle.c`` (plain C, fp64, POSIX threads); this
module compiles it with gcc on first use and marshals numpy arrays.  Each
function states the definition it follows; the citations are in ``oracle.c``.

Parity of every function here is pinned by ``tests/test_oracle_pins.py``
against exact integer arithmetic, exact rational arithmetic, closed forms,
invariants and library routines (numpy, torch), never against itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_gemm_bf16.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_bf16.restype = ctypes.c_int
            lib.oracle_gemm_w4a16.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_w4a16.restype = ctypes.c_int
            lib.oracle_dequant_w4.argtypes = [p, p, p, p, i64, i64, i64]
            lib.oracle_dequant_w4.restype = ctypes.c_int
            lib.oracle_round_to_bf16.argtypes = [p, p, i64]
            lib.oracle_round_to_bf16.restype = None
            lib.oracle_epilogue.argtypes = [ctypes.c_int, p, p, p, p, i64, i64]
            lib.oracle_epilogue.restype = ctypes.c_int
            lib.oracle_gemm_grouped.argtypes = [p, p, p, p, i64, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_grouped.restype = ctypes.c_int
            lib.oracle_gemm_mx.argtypes = [ctypes.c_int, p, p, ctypes.c_int, p, p, p, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm_mx.restype = ctypes.c_int
            lib.oracle_mx_decode.argtypes = [ctypes.c_int, p, p, i64]
            lib.oracle_mx_decode.restype = ctypes.c_int
            lib.oracle_hardware_threads.argtypes = []
            lib.oracle_hardware_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def _as(a, dtype, name):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"{name}: expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def gemm_bf16(A_bits: np.ndarray, B_bits: np.ndarray, threads: int | None = None) -> np.ndarray:
    """R[m,n] = sum_k A[m,k]*B[n,k] in fp64 (unrounded).

    A_bits: uint16 [M,K] bf16 bits; B_bits: uint16 [N,K] bf16 bits.
    """
    A = _as(A_bits, np.uint16, "A")
    B = _as(B_bits, np.uint16, "B")
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"shape mismatch {A.shape} x {B.shape}")
    M, K = A.shape
    N = B.shape[0]
    R = np.empty((M, N), dtype=np.float64)
    t = threads or hardware_threads()
    rc = _load().oracle_gemm_bf16(_ptr(A), _ptr(B), _ptr(R), M, N, K, K, K, t)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_bf16 returned {rc}")
    return R


def gemm_w4a16(A_bits: np.ndarray, Bq: np.ndarray, scales_bits: np.ndarray,
               zeros: np.ndarray, group: int, threads: int | None = None) -> np.ndarray:
    """R[m,n] = sum_k A[m,k]*(q[n,k]-z[n,k/g])*s[n,k/g] in fp64 (unrounded).

    A_bits uint16 [M,K]; Bq int32 [N,K/8]; scales_bits uint16 [N,K/g];
    zeros uint8 [N,K/g].
    """
    A = _as(A_bits, np.uint16, "A")
    Q = _as(Bq, np.int32, "Bq")
    S = _as(scales_bits, np.uint16, "scales")
    Z = _as(zeros, np.uint8, "zeros")
    M, K = A.shape
    N = Q.shape[0]
    if Q.shape != (N, K // 8) or S.shape != (N, K // group) or Z.shape != (N, K // group):
        raise ValueError("operand shapes do not match the stated W4A16 layout")
    R = np.empty((M, N), dtype=np.float64)
    t = threads or hardware_threads()
    rc = _load().oracle_gemm_w4a16(_ptr(A), _ptr(Q), _ptr(S), _ptr(Z), _ptr(R), M, N, K, group, K, t)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_w4a16 returned {rc}")
    return R


def gemm_bf16_bias(A_bits: np.ndarray, B_bits: np.ndarray, bias_bits: np.ndarray,
                   threads: int | None = None) -> np.ndarray:
    """R[m,n] = sum_k A[m,k]*B[n,k] + bias[n] in fp64 (unrounded); bias_bits uint16 [N]."""
    S = gemm_bf16(A_bits, B_bits, threads)
    b = _as(bias_bits, np.uint16, "bias")
    if b.shape != (S.shape[1],):
        raise ValueError("bias must have one entry per column of C")
    R = np.empty_like(S)
    rc = _load().oracle_epilogue(1, _ptr(S), None, _ptr(b), _ptr(R), S.shape[0], S.shape[1])
    if rc != 0:
        raise RuntimeError(f"oracle_epilogue returned {rc}")
    return R


def gemm_bf16_bias_act(A_bits: np.ndarray, B_bits: np.ndarray, bias_bits: np.ndarray, act: str,
                       threads: int | None = None) -> np.ndarray:
    """R[m,n] = act(sum_k A[m,k]*B[n,k] + bias[n]) in fp64 (unrounded), act
    "relu" (max(x, 0)), "silu" (x / (1 + e^-x)) or "gelu" (x/2 (1 + erf(x/sqrt 2)))."""
    S = gemm_bf16(A_bits, B_bits, threads)
    return bias_act(S, bias_bits, act)


def bias_act(S: np.ndarray, bias_bits: np.ndarray, act: str) -> np.ndarray:
    """act(S[m,n] + bias[n]) in fp64, S [M,N] fp64 (the epilogue alone, for pins)."""
    S = np.ascontiguousarray(S, dtype=np.float64)
    if S.ndim == 1:
        S = S.reshape(1, -1)
    b = _as(bias_bits, np.uint16, "bias")
    if b.shape != (S.shape[1],):
        raise ValueError("bias must have one entry per column")
    R = np.empty_like(S)
    rc = _load().oracle_epilogue({"relu": 3, "silu": 4, "gelu": 5}[act], _ptr(S), None, _ptr(b), _ptr(R),
                                 S.shape[0], S.shape[1])
    if rc != 0:
        raise RuntimeError(f"oracle_epilogue returned {rc}")
    return R


def gemm_bf16_silu_mul(A_bits: np.ndarray, B_bits: np.ndarray, threads: int | None = None) -> np.ndarray:
    """The fused gate/up projection: B_bits uint16 [2N,K] holds the gate rows
    0..N-1 and the up rows N..2N-1; R[m,n] = silu(g)*u in fp64 (unrounded)
    with g = sum_k A[m,k]*B[n,k], u = sum_k A[m,k]*B[N+n,k]."""
    B = _as(B_bits, np.uint16, "B")
    if B.ndim != 2 or B.shape[0] % 2:
        raise ValueError("B must hold 2N rows (gate, then up)")
    N = B.shape[0] // 2
    G = gemm_bf16(A_bits, B[:N], threads)
    U = gemm_bf16(A_bits, B[N:], threads)
    R = np.empty_like(G)
    rc = _load().oracle_epilogue(2, _ptr(G), _ptr(U), None, _ptr(R), G.shape[0], G.shape[1])
    if rc != 0:
        raise RuntimeError(f"oracle_epilogue returned {rc}")
    return R


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """silu(g)*u elementwise in fp64 (the epilogue alone, for pins)."""
    G = np.ascontiguousarray(g, dtype=np.float64)
    U = np.ascontiguousarray(u, dtype=np.float64)
    if G.shape != U.shape:
        raise ValueError("shape mismatch")
    R = np.empty_like(G)
    rc = _load().oracle_epilogue(2, _ptr(G), _ptr(U), None, _ptr(R), 1, G.size)
    if rc != 0:
        raise RuntimeError(f"oracle_epilogue returned {rc}")
    return R


def gemm_grouped(A_bits: np.ndarray, B_bits: np.ndarray, ends: np.ndarray,
                 threads: int | None = None) -> np.ndarray:
    """The grouped (MoE) GEMM in fp64: A_bits uint16 [M,K] stacked token rows,
    B_bits uint16 [G,N,K] per-expert weights, ends int32 [G] cumulative row
    ends; R[m,n] = sum_k A[m,k]*B[g,n,k] for the expert g owning row m, 0 for
    rows past ends[-1]."""
    A = _as(A_bits, np.uint16, "A")
    B = _as(B_bits, np.uint16, "B")
    E = _as(ends, np.int32, "ends")
    if A.ndim != 2 or B.ndim != 3 or A.shape[1] != B.shape[2] or E.shape != (B.shape[0],):
        raise ValueError("shape mismatch for the grouped GEMM")
    M, K = A.shape
    G, N, _ = B.shape
    R = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_grouped(_ptr(A), _ptr(B), _ptr(E), _ptr(R), G, M, N, K,
                                     threads or hardware_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_grouped returned {rc}")
    return R


MX_FORMATS = {"e4m3": 0, "e2m1": 1}


def gemm_mx(A: np.ndarray, SA: np.ndarray, B: np.ndarray, SB: np.ndarray, fmt_a: str = "e4m3",
            fmt_b: str = "e4m3", threads: int | None = None) -> np.ndarray:
    """The block-scaled (MX) GEMM in fp64 (unrounded):
    R[m,n] = sum_k a[m,k] 2^(SA[m,k/32]-127) * b[n,k] 2^(SB[n,k/32]-127).

    A: uint8 E4M3 codes [M,K] or packed E2M1 [M,K/2] (element k in bits
    4*(k%2)..); B likewise [N,K] / [N,K/2]; SA uint8 [M,K/32], SB uint8
    [N,K/32] E8M0 codes.
    """
    fa, fb = MX_FORMATS[fmt_a], MX_FORMATS[fmt_b]
    A = _as(A, np.uint8, "A")
    B = _as(B, np.uint8, "B")
    SA = _as(SA, np.uint8, "SA")
    SB = _as(SB, np.uint8, "SB")
    M, N = A.shape[0], B.shape[0]
    K = A.shape[1] * (2 if fa else 1)
    if B.shape[1] * (2 if fb else 1) != K or K % 32 or SA.shape != (M, K // 32) or SB.shape != (N, K // 32):
        raise ValueError("MX operand shapes do not match")
    R = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_mx(fa, _ptr(A), _ptr(SA), fb, _ptr(B), _ptr(SB), _ptr(R), M, N, K,
                                threads or hardware_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_mx returned {rc}")
    return R


def mx_decode(codes: np.ndarray, kind: str) -> np.ndarray:
    """Values of MX codes (one per byte): kind "e4m3", "e2m1" (low nibble) or "e8m0"."""
    c = _as(codes, np.uint8, "codes")
    out = np.empty(c.shape, dtype=np.float64)
    rc = _load().oracle_mx_decode({"e4m3": 0, "e2m1": 1, "e8m0": 2}[kind], _ptr(c), _ptr(out), c.size)
    if rc != 0:
        raise RuntimeError(f"oracle_mx_decode returned {rc}")
    return out


def dequant_w4(Bq: np.ndarray, scales_bits: np.ndarray, zeros: np.ndarray, group: int) -> np.ndarray:
    """W[n,k] = (q[n,k] - z[n,k/g]) * s[n,k/g] as fp64 [N,K]."""
    Q = _as(Bq, np.int32, "Bq")
    S = _as(scales_bits, np.uint16, "scales")
    Z = _as(zeros, np.uint8, "zeros")
    N, words = Q.shape
    K = words * 8
    W = np.empty((N, K), dtype=np.float64)
    rc = _load().oracle_dequant_w4(_ptr(Q), _ptr(S), _ptr(Z), _ptr(W), N, K, group)
    if rc != 0:
        raise RuntimeError(f"oracle_dequant_w4 returned {rc}")
    return W


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits (uint16), round to nearest, ties to even, one rounding."""
    X = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(X.shape, dtype=np.uint16)
    _load().oracle_round_to_bf16(_ptr(X), _ptr(out), X.size)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bits -> fp64 values (exact widening; the bits are the top of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def within_tolerance(out: np.ndarray, ref: np.ndarray, rms_ref: float | None = None):
    """Per-element check |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).

    rms(ref) is taken over all entries of ``ref`` unless the caller passes the
    rms of the full output (for sampled checks).  Returns (ok_mask, rms).
    """
    ref = np.asarray(ref, dtype=np.float64)
    out = np.asarray(out, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if rms_ref is None else float(rms_ref)
    ok = np.abs(out - ref) <= 1e-2 * np.abs(ref) + 1e-2 * rms
    return ok, rms
