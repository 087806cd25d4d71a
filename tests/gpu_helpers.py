"""Helpers shared by the GPU parity tests (host <-> device marshalling and the
oracle comparisons).  Inputs come from dense_bit_weight_gb300.synth; expected
values come only from the oracle."""
import numpy as np

import oracle
from dense_bit_weight_gb300 import synth


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_raw(x: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host_bits(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_inputs(M, N, K, seed=0, kind="normal"):
    """A [M,K], B [N,K] bf16 bits: N(0,1) and N(0, 1/K) (std 1/sqrt(K)), or
    integers uniform in [-4, 4]."""
    if kind == "int":
        return (synth.bf16_int_uniform((M, K), -4, 4, seed, synth.STREAM_A_INT),
                synth.bf16_int_uniform((N, K), -4, 4, seed, synth.STREAM_B_INT))
    return (synth.bf16_normal((M, K), 1.0, seed, synth.STREAM_A),
            synth.bf16_normal((N, K), K ** -0.5 if K else 1.0, seed, synth.STREAM_B))


def assert_close(out_bits: np.ndarray, ref: np.ndarray, rms=None, what=""):
    out = oracle.bf16_bits_to_f64(out_bits)
    ok, r = oracle.within_tolerance(out, ref, rms)
    if not ok.all():
        bad = np.argwhere(~ok)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} out of tolerance; first {i}: "
                             f"out={out[i]!r} ref={ref[i]!r} rms={r:.4g}")


def assert_exact(out_bits: np.ndarray, ref: np.ndarray, what=""):
    want = oracle.round_to_bf16(ref)
    if not np.array_equal(out_bits, want):
        bad = np.argwhere(out_bits != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {want.size} differ; first {i}: "
                             f"got {out_bits[i]:#06x} want {want[i]:#06x} (ref {ref[i]!r})")


def sample_rows(M, k=4, seed=0):
    rng = np.random.default_rng(seed)
    pick = {0, M - 1} | set(rng.integers(0, M, size=k).tolist())
    return np.array(sorted(pick))
