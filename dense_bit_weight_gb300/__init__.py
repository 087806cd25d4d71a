"""GB300-native projection GEMM: C[M,N] = A[M,K] . B[N,K]^T (bf16, and W4A16).

The compute path is the C-ABI library ``libdbw_gemm.so`` (hand-written sm_103a
CUDA); ``dense_bit_weight_gb300.gemm`` is its thin ctypes binding.  Importing
this package does not load the library; the binding raises if it is missing.
"""
__all__ = ["gemm", "synth", "build"]
