"""Thin ctypes binding of libdbw_gemm.so (the C ABI in include/dbw_gemm.h).

Argument marshalling only: torch tensors become device pointers, sizes and
the current CUDA stream handle; every step of the computation runs in the
library's kernels.  Importing this module loads the library and raises
ImportError when it has not been built -- there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libdbw_gemm.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
lib = ctypes.CDLL(_LIB_PATH)

GEMM_OK = 0
STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_NULL", 2: "GEMM_ERR_SHAPE", 3: "GEMM_ERR_LD",
          4: "GEMM_ERR_ALIGN", 5: "GEMM_ERR_GROUP", 6: "GEMM_ERR_CUDA",
          7: "GEMM_ERR_DEVICE_TIMEOUT", 8: "GEMM_ERR_ARCH", 9: "GEMM_ERR_ALIAS",
          10: "GEMM_ERR_VARIANT", 11: "GEMM_ERR_EPILOGUE"}
VARIANT = {"auto": 0, "gemv": 1, "skinny": 2, "prefill": 3, "zero": 4, "register": 5, "fragment": 6,
           "groupwise": 7, "block_scaled": 8, "pair": 9, "band": 10}
VARIANT_NAME = {v: k for k, v in VARIANT.items()}

EXPORTS = ["gemm_bf16", "gemm_w4a16", "gemm_bf16_ex", "gemm_w4a16_ex", "gemm_bf16_plan",
           "gemm_w4a16_plan", "gemm_last_device_error", "gemm_status_string", "gemm_shutdown",
           "gemm_debug_inject_timeout", "gemm_bf16_noalloc", "gemm_bf16_noalloc_last_error", "gemm_bf16_fused", "gemm_bf16_fused_ex",
           "gemm_bf16_grouped", "gemm_bf16_fused_plan", "gemm_mxfp8", "gemm_mxfp4", "gemm_mx_plan"]


class gemm_plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("kernels", ctypes.c_int), ("grid", ctypes.c_int),
                ("split", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("stages", ctypes.c_int), ("reserved", ctypes.c_int)]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["variant_name"] = VARIANT_NAME.get(self.variant, "?")
        return d


_p, _i64, _i = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
lib.gemm_bf16.argtypes = [_p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _p]
lib.gemm_bf16_ex.argtypes = lib.gemm_bf16.argtypes + [_i]
lib.gemm_bf16_fused_ex.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i, _p, _i]
lib.gemm_bf16_fused_ex.restype = _i
lib.gemm_bf16_grouped.argtypes = [_p, _p, _p, _p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _p]
lib.gemm_bf16_grouped.restype = _i
lib.gemm_bf16_noalloc.argtypes = lib.gemm_bf16.argtypes
lib.gemm_bf16_noalloc.restype = _i
lib.gemm_bf16_noalloc_last_error.argtypes = []
lib.gemm_bf16_noalloc_last_error.restype = _i
lib.gemm_mxfp8.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.gemm_mxfp8.restype = _i
lib.gemm_mxfp4.argtypes = lib.gemm_mxfp8.argtypes
lib.gemm_mxfp4.restype = _i
lib.gemm_mx_plan.argtypes = [_i64, _i64, _i64, _i, _i, ctypes.POINTER(gemm_plan)]
lib.gemm_mx_plan.restype = _i
lib.gemm_w4a16.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _i64, _p]
lib.gemm_w4a16_ex.argtypes = lib.gemm_w4a16.argtypes + [_i]
lib.gemm_bf16_plan.argtypes = [_i64, _i64, _i64, _i, _i, ctypes.POINTER(gemm_plan)]
lib.gemm_w4a16_plan.argtypes = [_i64, _i64, _i64, _i64, _i, _i, ctypes.POINTER(gemm_plan)]
lib.gemm_bf16_fused_plan.argtypes = [_i64, _i64, _i64, _i, _i, _i, ctypes.POINTER(gemm_plan)]
lib.gemm_last_device_error.argtypes = []
lib.gemm_status_string.argtypes = [_i]
lib.gemm_status_string.restype = ctypes.c_char_p
lib.gemm_debug_inject_timeout.argtypes = [_i]
lib.gemm_debug_inject_timeout.restype = _i
lib.gemm_shutdown.argtypes = []
lib.gemm_shutdown.restype = None
for _f in ("gemm_bf16", "gemm_bf16_ex", "gemm_w4a16", "gemm_w4a16_ex", "gemm_bf16_plan",
           "gemm_w4a16_plan", "gemm_bf16_fused_plan", "gemm_last_device_error"):
    getattr(lib, _f).restype = _i


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({gemm_status_string(status)})")


def _check(rc: int, where: str):
    if rc != GEMM_OK:
        raise GemmError(rc, where)


def gemm_status_string(status: int) -> str:
    return lib.gemm_status_string(int(status)).decode()


def gemm_last_device_error() -> int:
    return int(lib.gemm_last_device_error())


def gemm_bf16_noalloc_last_error() -> int:
    """The watchdog word of gemm_bf16_noalloc (read and cleared)."""
    return int(lib.gemm_bf16_noalloc_last_error())


def gemm_debug_inject_timeout(enable: bool) -> bool:
    """Test hook: make the tcgen05 kernels' bounded waits expire (see the header)."""
    return bool(lib.gemm_debug_inject_timeout(1 if enable else 0))


def gemm_shutdown() -> None:
    lib.gemm_shutdown()


def _variant(v) -> int:
    return VARIANT[v] if isinstance(v, str) else int(v)


def gemm_bf16_plan(M: int, N: int, K: int, variant="auto", num_sms: int = 0) -> dict:
    out = gemm_plan()
    _check(lib.gemm_bf16_plan(M, N, K, _variant(variant), num_sms, ctypes.byref(out)), "gemm_bf16_plan")
    return out.as_dict()


def gemm_bf16_fused_plan(M: int, N: int, K: int, epilogue="silu_mul", variant="auto", num_sms: int = 0) -> dict:
    """Plan of gemm_bf16_fused (N = columns of C)."""
    epi = EPILOGUE[epilogue] if isinstance(epilogue, str) else int(epilogue)
    out = gemm_plan()
    _check(lib.gemm_bf16_fused_plan(M, N, K, epi, _variant(variant), num_sms, ctypes.byref(out)),
           "gemm_bf16_fused_plan")
    return out.as_dict()


def gemm_w4a16_plan(M: int, N: int, K: int, group: int, variant="auto", num_sms: int = 0) -> dict:
    out = gemm_plan()
    _check(lib.gemm_w4a16_plan(M, N, K, group, _variant(variant), num_sms, ctypes.byref(out)),
           "gemm_w4a16_plan")
    return out.as_dict()


# --------------------------------------------------------------- torch layer

def _stream_handle(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _same_cuda_device(ref, *tensors):
    """Every tensor (None skipped) must be a CUDA tensor on ref's device: the C
    calls take raw device addresses and cannot tell host memory apart."""
    for name, t in tensors:
        if t is not None and (not t.is_cuda or t.device != ref.device):
            raise ValueError(f"{name} must be a CUDA tensor on {ref.device}")


def _row_major_2d(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit stride along its last dimension")
    return t.stride(0)


def gemm_bf16(A, B, C=None, stream=None, variant="auto"):
    """C[M,N] = A[M,K] @ B[N,K]^T on the device (bf16 in, fp32 accumulate, bf16 out).

    A and B are CUDA bf16 tensors with unit stride along K; C (optional) is a
    CUDA bf16 [M,N] tensor with unit stride along N.  Runs on ``stream`` (the
    current torch stream by default) without synchronising.  Returns C.
    """
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError(f"K mismatch: {A.shape} vs {B.shape}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or tuple(C.shape) != (M, N):
        raise ValueError("C must be bfloat16 [M,N]")
    _same_cuda_device(A, ("B", B), ("C", C))
    lda, ldb, ldc = _row_major_2d(A, "A"), _row_major_2d(B, "B"), _row_major_2d(C, "C")
    rc = lib.gemm_bf16_ex(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, lda, ldb, ldc,
                          _stream_handle(stream), _variant(variant))
    _check(rc, "gemm_bf16")
    return C


EPILOGUE = {"none": 0, "bias": 1, "silu_mul": 2, "bias_relu": 3, "bias_silu": 4, "bias_gelu": 5}


def gemm_bf16_fused(A, B, bias=None, C=None, epilogue="bias", stream=None, variant="auto"):
    """gemm_bf16 with a fused epilogue (applied in fp32 to the full K sum).

    epilogue "bias": C[m,n] = (A @ B^T)[m,n] + bias[n] (bias bf16 [N]);
    "bias_relu" / "bias_silu" / "bias_gelu": the activation of that sum.
    epilogue "silu_mul": B is the fused gate/up weight [2N,K] (gate rows, then
    up rows) and C[m,n] = silu(g) * u with g, u the two halves of A @ B^T.
    Returns C bf16 [M,N].
    """
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if not (A.is_cuda and B.is_cuda):
        raise ValueError("A and B must be CUDA tensors")
    epi = EPILOGUE[epilogue] if isinstance(epilogue, str) else int(epilogue)
    M, K = A.shape
    NB, K2 = B.shape
    if K != K2:
        raise ValueError(f"K mismatch: {A.shape} vs {B.shape}")
    if epi == 2 and NB % 2:
        raise ValueError("silu_mul: B must hold 2N rows (gate, then up)")
    N = NB // 2 if epi == 2 else NB
    if bias is not None and (bias.dtype != torch.bfloat16 or not bias.is_cuda or tuple(bias.shape) != (N,)
                             or bias.stride(0) != 1):
        raise ValueError("bias must be a contiguous CUDA bfloat16 [N] tensor")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or tuple(C.shape) != (M, N):
        raise ValueError("C must be bfloat16 [M,N]")
    _same_cuda_device(A, ("B", B), ("C", C), ("bias", bias))
    lda, ldb, ldc = _row_major_2d(A, "A"), _row_major_2d(B, "B"), _row_major_2d(C, "C")
    rc = lib.gemm_bf16_fused_ex(A.data_ptr(), B.data_ptr(), bias.data_ptr() if bias is not None else None,
                                C.data_ptr(), M, N, K, lda, ldb, ldc, epi, _stream_handle(stream),
                                _variant(variant))
    _check(rc, "gemm_bf16_fused")
    return C


def gemm_bf16_grouped(A, B, ends, C=None, stream=None):
    """The grouped (MoE) GEMM: expert g's token rows ends[g-1]..ends[g]-1 of A
    [M,K] times its weights B[g] ([G,N,K]); C [M,N] rows past ends[-1] are not
    written.  ends: CUDA int32 [G] cumulative row ends.  Returns C."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if B.dim() != 3 or not B.is_contiguous() or ends.dtype != torch.int32 or ends.dim() != 1 \
            or not ends.is_cuda or not ends.is_contiguous():
        raise ValueError("B must be a contiguous [G,N,K] tensor and ends a contiguous CUDA int32 [G] tensor")
    M, K = A.shape
    G, N, K2 = B.shape
    if K != K2 or ends.shape[0] != G:
        raise ValueError("shape mismatch")
    if C is None:
        C = torch.zeros((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or tuple(C.shape) != (M, N):
        raise ValueError("C must be bfloat16 [M,N]")
    _same_cuda_device(A, ("A", A), ("B", B), ("C", C), ("ends", ends))
    lda, ldc = _row_major_2d(A, "A"), _row_major_2d(C, "C")
    rc = lib.gemm_bf16_grouped(A.data_ptr(), B.data_ptr(), C.data_ptr(), ends.data_ptr(), G, M, N, K,
                               lda, K, ldc, _stream_handle(stream))
    _check(rc, "gemm_bf16_grouped")
    return C


def gemm_w4a16(A, Bq, scales, zeros, group: int, C=None, stream=None, variant="auto"):
    """C[M,N] = A[M,K] @ W[N,K]^T with W = (q - z) * s, q packed 8 per int32 along K.

    A bf16 [M,K]; Bq int32 [N,K/8]; scales bf16 [N,K/group]; zeros uint8
    [N,K/group]; all contiguous CUDA tensors.  Returns C bf16 [M,N].
    """
    import torch
    M, K = A.shape
    N = Bq.shape[0]
    for t, name, dt in ((A, "A", torch.bfloat16), (Bq, "Bq", torch.int32),
                        (scales, "scales", torch.bfloat16), (zeros, "zeros", torch.uint8)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    if tuple(Bq.shape) != (N, K // 8) or tuple(scales.shape) != (N, K // group) \
            or tuple(zeros.shape) != (N, K // group):
        raise ValueError("W4A16 operand shapes do not match")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or tuple(C.shape) != (M, N) or not C.is_contiguous():
        raise ValueError("C must be a contiguous bfloat16 [M,N] tensor")
    _same_cuda_device(A, ("Bq", Bq), ("scales", scales), ("zeros", zeros), ("C", C))
    rc = lib.gemm_w4a16_ex(A.data_ptr(), Bq.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                           C.data_ptr(), M, N, K, group, _stream_handle(stream), _variant(variant))
    _check(rc, "gemm_w4a16")
    return C


MX_FMT = {"e4m3": 0, "e2m1": 1}


def gemm_mx_plan(M: int, N: int, K: int, fmt="e4m3", num_sms: int = 0) -> dict:
    out = gemm_plan()
    _check(lib.gemm_mx_plan(M, N, K, MX_FMT[fmt] if isinstance(fmt, str) else int(fmt), num_sms,
                            ctypes.byref(out)), "gemm_mx_plan")
    return out.as_dict()


def gemm_mx(A, SA, B, SB, fmt="e4m3", C=None, stream=None):
    """The block-scaled (MX) GEMM: C[M,N] bf16 = sum_k a 2^(SA-127) * b 2^(SB-127).

    fmt "e4m3": A uint8 [M,K], B uint8 [N,K] (E4M3 codes); fmt "e2m1": A
    uint8 [M,K/2], B uint8 [N,K/2] (packed, low nibble first).  SA uint8
    [M,K/32], SB uint8 [N,K/32] (E8M0 codes).  All contiguous CUDA tensors.
    """
    import torch
    f = MX_FMT[fmt]
    M, N = A.shape[0], B.shape[0]
    K = A.shape[1] * (2 if f else 1)
    for t, name in ((A, "A"), (SA, "SA"), (B, "B"), (SB, "SB")):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D CUDA uint8 tensor")
    if B.shape[1] * (2 if f else 1) != K or tuple(SA.shape) != (M, K // 32) or tuple(SB.shape) != (N, K // 32):
        raise ValueError("MX operand shapes do not match")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if C.dtype != torch.bfloat16 or tuple(C.shape) != (M, N) or not C.is_contiguous():
        raise ValueError("C must be a contiguous bfloat16 [M,N] tensor")
    _same_cuda_device(A, ("SA", SA), ("B", B), ("SB", SB), ("C", C))
    fn = lib.gemm_mxfp8 if f == 0 else lib.gemm_mxfp4
    _check(fn(A.data_ptr(), SA.data_ptr(), B.data_ptr(), SB.data_ptr(), C.data_ptr(), M, N, K,
              _stream_handle(stream)), "gemm_mx" + ("fp8" if f == 0 else "fp4"))
    return C


# --------------------------------------------------------------- raw pointers

def gemm_bf16_ptr(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                  stream: int = 0, variant="auto") -> int:
    """The C call on raw device addresses; returns the gemm_status."""
    return int(lib.gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, ctypes.c_void_p(stream),
                                _variant(variant)))


def gemm_bf16_fused_ptr(A: int, B: int, bias: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                        ldc: int, epilogue: int, stream: int = 0, variant="auto") -> int:
    """gemm_bf16_fused_ex on raw device addresses (bias 0 = NULL); returns the gemm_status."""
    return int(lib.gemm_bf16_fused_ex(A, B, bias or None, C, M, N, K, lda, ldb, ldc, epilogue,
                                      ctypes.c_void_p(stream), _variant(variant)))


def gemm_bf16_noalloc_ptr(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int,
                          ldc: int, stream: int = 0) -> int:
    """gemm_bf16_noalloc on raw device addresses (allocates nothing); returns the gemm_status."""
    return int(lib.gemm_bf16_noalloc(A, B, C, M, N, K, lda, ldb, ldc, ctypes.c_void_p(stream)))


def gemm_w4a16_ptr(A: int, Bq: int, scales: int, zeros: int, C: int, M: int, N: int, K: int,
                   group: int, stream: int = 0, variant="auto") -> int:
    return int(lib.gemm_w4a16_ex(A, Bq, scales, zeros, C, M, N, K, group, ctypes.c_void_p(stream),
                                 _variant(variant)))


def gemm_mx_ptr(fmt: str, A: int, SA: int, B: int, SB: int, C: int, M: int, N: int, K: int,
                stream: int = 0) -> int:
    """gemm_mxfp8 / gemm_mxfp4 on raw device addresses; returns the gemm_status."""
    fn = lib.gemm_mxfp8 if MX_FMT[fmt] == 0 else lib.gemm_mxfp4
    return int(fn(A, SA, B, SB, C, M, N, K, ctypes.c_void_p(stream)))
