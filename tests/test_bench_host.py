"""Host-side pieces of bench.py (no GPU): the packing of the end-to-end
step's copies, the traffic table's keys, and the reference arm's JSON line."""
import importlib.util
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_pack_e2e_views_and_contents(bench):
    torch = pytest.importorskip("torch")
    gen = torch.Generator().manual_seed(3)
    items = []
    for (M, N, K) in ((1, 24, 16), (3, 40, 8), (8, 16, 64), (5, 8, 24)):
        items.append(dict(M=M, N=N, K=K, A=torch.randn((M, K), generator=gen).to(torch.bfloat16),
                          B=None, C=torch.empty((M, N), dtype=torch.bfloat16)))
    host_a, dev_a, host_c, dev_c, packed = bench.pack_e2e(torch, items, "cpu", pin=False)
    assert len(packed) == len(items)
    # the host buffer holds every item's activations; one copy moves them all
    dev_a.copy_(host_a)
    for it, p in zip(items, packed):
        assert p["A"].shape == (it["M"], it["K"]) and p["C"].shape == (it["M"], it["N"])
        assert p["A"].is_contiguous() and p["C"].is_contiguous()
        assert p["A"].data_ptr() % 16 == 0 and p["C"].data_ptr() % 16 == 0
        assert p["A"].untyped_storage().data_ptr() == dev_a.untyped_storage().data_ptr()
        assert p["C"].untyped_storage().data_ptr() == dev_c.untyped_storage().data_ptr()
        assert torch.equal(p["A"], it["A"])
        assert (p["M"], p["N"], p["K"]) == (it["M"], it["N"], it["K"])
    # outputs written through the views come back with one copy, at disjoint places
    for i, p in enumerate(packed):
        p["C"].fill_(float(i + 1))
    host_c.copy_(dev_c)
    seen = set()
    for i, p in enumerate(packed):
        off = (p["C"].data_ptr() - dev_c.data_ptr()) // 2
        n = p["M"] * p["N"]
        block = host_c[off:off + n].float().numpy()
        assert np.all(block == i + 1)
        assert not (set(range(off, off + n)) & seen)
        seen |= set(range(off, off + n))


def test_traffic_table_covers_the_decode_step(bench):
    assert set(bench.TRAFFIC_BYTES) == set(bench.DECODE)
    for (M, N, K), b in bench.TRAFFIC_BYTES.items():
        alg = bench.bytes_bf16(M, N, K)
        assert 0.9 * alg < b < 1.1 * alg        # measured DRAM bytes near the algorithmic count
    assert len(bench.kernel_sources_sha256()) == 64


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--ref-step-seconds", "0.2"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
