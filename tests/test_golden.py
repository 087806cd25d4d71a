"""The oracle against hand-worked examples stored under tests/golden/."""
import os

import numpy as np

import oracle
from dense_bit_weight_gb300 import synth

HERE = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.txt")


def _cases():
    cases, cur = [], None
    for line in open(HERE):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = (s.strip() for s in line.split("=", 1))
        if k == "kind":
            cur = {"kind": v}
            cases.append(cur)
        else:
            cur[k] = v
    return cases


def _floats(s):
    return np.array([float(x) for x in s.split(",")])


def _bf16(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def test_hand_examples():
    cases = _cases()
    assert len(cases) == 2
    for c in cases:
        M, N, K = int(c["M"]), int(c["N"]), int(c["K"])
        if c["kind"] == "bf16":
            A = _bf16(_floats(c["A"]).reshape(M, K))
            B = _bf16(_floats(c["B"]).reshape(N, K))
            R = oracle.gemm_bf16(A, B)
        else:
            g = int(c["group"])
            A = _bf16(np.ones((M, K)))
            Bq = np.full((N, K // 8), int(c["Bq_word"], 16), dtype=np.uint32).view(np.int32)
            Z = _floats(c["zeros"]).astype(np.uint8).reshape(N, K // g)
            S = _bf16(_floats(c["scales"]).reshape(N, K // g))
            R = oracle.gemm_w4a16(A, Bq, S, Z, g)
        assert np.array_equal(R, _floats(c["C"]).reshape(M, N)), c["kind"]
