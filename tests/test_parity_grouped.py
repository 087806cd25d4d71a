"""GPU parity of gemm_bf16_grouped (the mixture-of-experts GEMM) against the fp64 oracle.

Uniform, ragged, empty and skewed expert loads, offsets that end before M
(rows past the last expert are not written) and out-of-range offsets (which
the kernel clamps), compared element by element, and the three loads the
bench times at full size (8 experts x 512 tokens and a ragged 16-expert load
with empty experts, N = K = 4096; 128 experts x 4 tokens, N = 1536, K = 2048),
also every element; integer-valued inputs must
match bit for bit, N(0,1) inputs satisfy |out - ref| <= 1e-2*|ref| + 1e-2*rms(ref).
"""
import numpy as np
import pytest

import oracle
from dense_bit_weight_gb300 import synth
from gpu_helpers import assert_close, assert_exact, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import torch
    from dense_bit_weight_gb300 import gemm
    torch.cuda.init()
    yield gemm
    assert gemm.gemm_last_device_error() == 0


def operands(M, G, N, K, kind, seed):
    if kind == "int":
        A = synth.bf16_int_uniform((M, K), -4, 4, seed, synth.STREAM_A_INT)
        B = synth.bf16_int_uniform((G * N, K), -4, 4, seed, synth.STREAM_B_INT)
    else:
        A = synth.bf16_normal((M, K), 1.0, seed, synth.STREAM_A)
        B = synth.bf16_normal((G * N, K), K ** -0.5, seed, synth.STREAM_B)
    return A, B.reshape(G, N, K)


def run(g, A, B, ends, M, N):
    import torch
    C = torch.full((M, N), -7.0, dtype=torch.bfloat16, device="cuda")   # marks rows it must not write
    g.gemm_bf16_grouped(dev_bf16(A), dev_bf16(B.reshape(-1, B.shape[2])).reshape(B.shape),
                        torch.tensor(ends, dtype=torch.int32, device="cuda"), C=C)
    return host_bits(C)


CASES = [  # (expert token counts, N, K, spare rows past the last expert)
    ([256, 256, 256, 256], 512, 512, 0),           # uniform
    ([1, 0, 300, 17, 0, 129, 64, 2], 384, 256, 5),  # ragged with empty experts
    ([0, 0, 0, 1000], 264, 1024, 3),                # all tokens on one expert
    ([3] * 64, 256, 128, 0),                        # many small experts (decode-like)
    ([130], 4104, 72, 0),                           # one expert = the plain GEMM, ragged N
    ([700, 0, 300, 513], 264, 520, 7),              # CTA pairs (>= 256 tokens per expert on average):
                                                    # partial m-tiles, an empty expert, ragged N and K
    # the bench's loads, full size
    ([512] * 8, 4096, 4096, 0),
    ([1024, 0, 512, 37, 0, 800, 256, 1, 600, 0, 300, 64, 200, 150, 100, 52], 4096, 4096, 0),
    ([4] * 128, 1536, 2048, 0),
]


@pytest.mark.parametrize("sizes,N,K,spare", CASES)
@pytest.mark.parametrize("kind", ["int", "normal"])
def test_grouped(g, sizes, N, K, spare, kind):
    G = len(sizes)
    ends = np.cumsum(sizes).astype(np.int32)
    M = int(ends[-1]) + spare
    A, B = operands(M, G, N, K, kind, seed=G + N)
    C = run(g, A, B, ends, M, N)
    last = int(ends[-1])
    ref = oracle.gemm_grouped(A, B, ends)[:last]
    (assert_exact if kind == "int" else assert_close)(C[:last], ref, what=f"grouped {sizes[:6]} N={N} K={K}")
    assert (C[last:] == 0xC0E0).all()   # -7.0 untouched past the last expert


def test_out_of_range_offsets_are_clamped(g):
    M, N, K = 200, 256, 256
    raw = np.array([50, 30, 120, 500], dtype=np.int32)   # decreasing step, end past M
    A, B = operands(M, 4, N, K, "int", seed=3)
    C = run(g, A, B, raw, M, N)
    ends = np.minimum(np.maximum.accumulate(raw), M).astype(np.int32)   # the documented clamp
    assert_exact(C, oracle.gemm_grouped(A, B, ends), what="clamped offsets")


def test_router_offsets_written_by_the_previous_kernel(g):
    # the offsets are produced on the stream right before the GEMM (as a
    # router would), with no host synchronisation in between
    import torch
    M, N, K, G = 512, 256, 512, 8
    A, B = operands(M, G, N, K, "int", seed=4)
    counts = torch.tensor([64, 0, 100, 36, 200, 0, 12, 100], dtype=torch.int32, device="cuda")
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    dA, dB = dev_bf16(A), dev_bf16(B.reshape(-1, K)).reshape(G, N, K)
    ends = torch.cumsum(counts, 0, dtype=torch.int32)
    g.gemm_bf16_grouped(dA, dB, ends, C=C)
    want = oracle.gemm_grouped(A, B, np.cumsum(counts.cpu().numpy()).astype(np.int32))
    assert_exact(host_bits(C), want, what="router offsets")
