"""Benchmark of the projection GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass over the decode-projection workload: C = A . B^T for
M in {1, 8, 32, 128} tokens against three bf16 weight matrices of
Qwen3-8B-like dimensions (qkv 6144x4096, o 4096x4096, fused gate/up
24576x4096), twelve GEMMs per step.  Every GEMM has its own weight copy
(1.14 GB streamed per step, nine times the L2), so weights come from HBM.
The metric is algorithmic HBM bytes, 2*(M*K + N*K + M*N) per GEMM, divided
by device time (CUDA events on the launching stream).

The JSON line also carries:
  roofline      the dominant kernel's algorithmic GB/s (bytes / its own
                event-timed launch durations) against the measured HBM peak
  e2e           the same metric through the public call with host buffers:
                each step copies its activations host->device (pinned) and
                its outputs device->host; weights stay resident
  cpu_baseline  the fp64 CPU oracle on this host, on a bounded sample
  sweeps        prefill (TFLOP/s), down-projection and W4A16 (GB/s) shapes, and the
                fused gate/up projection with the SiLU-mul epilogue (decode GB/s,
                prefill TFLOP/s), the grouped (MoE) GEMM, and W4A16 at
                prefill-size token counts (TFLOP/s)
                and the block-scaled (MX) GEMMs, E4M3 and E2M1 (TFLOP/s)
  clocks        nvidia-smi samples taken during the timed region

--impl reference times the oracle (the method's plain definition on the
host cores) on a sample of the same workload.  Multi-GPU runs are replicas:
each rank runs the whole step on its own GPU; value sums over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (prefill) & HBM GB/s (decode), % of GB300 roofline"
DECODE = [(M, N, 4096) for M in (1, 8, 32, 128) for N in (6144, 4096, 24576)]
DOWN = [(M, 4096, 12288) for M in (1, 16, 64, 128, 512)]
PREFILL = [(M, N, K) for M in (1024, 4096, 16384)
           for (N, K) in ((4096, 4096), (6144, 4096), (24576, 4096), (4096, 12288), (8192, 8192))]
W4 = [(M, N, K) for M in (1, 16, 64, 128)
      for (N, K) in ((7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408))]
# W4A16 at prefill-size token counts (TFLOP/s)
W4_PREFILL = [(1024, 34816, 5120), (4096, 34816, 5120), (4096, 5120, 17408)]
# fused gate/up projection with the SiLU-mul epilogue (C has N = 12288 columns, B 2N rows)
GATE_UP_DECODE = [(M, 12288, 4096) for M in (1, 8, 32, 128)]
GATE_UP_PREFILL = [(M, 12288, 4096) for M in (1024, 4096)]
# grouped (MoE) GEMM: (name, expert token counts, N, K); ragged includes empty experts
GROUPED = [("uniform 8 experts", [512] * 8, 4096, 4096),
           ("ragged 16 experts", [1024, 0, 512, 37, 0, 800, 256, 1, 600, 0, 300, 64, 200, 150, 100, 52], 4096, 4096),
           ("decode MoE 128 experts", [4] * 128, 1536, 2048)]
# block-scaled (MX) GEMMs: the prefill shapes, plus the pages' MXFP shapes
# (32 x 4096 x 4096 for MXFP8, 32 x 14336 x 4096 for MXFP4)
MX_SHAPES = [(32, 4096, 4096), (32, 14336, 4096)] + PREFILL
# dense tensor peaks per format relative to bf16 (nominal GB300 figures:
# bf16 2.25, fp8 4.5, fp4 13.5 PFLOP/s); the bench scales the measured bf16 peak
MX_PEAK_RATIO = {"e4m3": 2.0, "e2m1": 6.0}
WORKLOAD = ("decode projections, Qwen3-8B-like dims: bf16 A[M,4096], M in {1,8,32,128}, "
            "B in {qkv 6144x4096, o 4096x4096, gate/up 24576x4096}, fp32 accumulate, bf16 out")


# DRAM bytes (read + write) per launch of each decode GEMM, from one ncu pass
# per shape (profiles/decode_step_dram_traffic.md) over the sources of the
# decode step's kernels and their planner (DECODE_KERNEL_SOURCES) with this
# SHA-256; reported only while those sources are unchanged.
TRAFFIC_SOURCES_SHA256 = "66104083d2303030a902e631ecd228c56aee28307a799c6879a0ec29ee519724"
TRAFFIC_BYTES = {(1, 4096, 4096): 33.57e6, (1, 6144, 4096): 50.38e6, (1, 24576, 4096): 204.19e6,
                 (8, 4096, 4096): 33.66e6, (8, 6144, 4096): 50.43e6, (8, 24576, 4096): 204.27e6,
                 (32, 4096, 4096): 33.91e6, (32, 6144, 4096): 50.69e6, (32, 24576, 4096): 204.42e6,
                 (128, 4096, 4096): 34.70e6, (128, 6144, 4096): 51.54e6, (128, 24576, 4096): 205.29e6}


DECODE_KERNEL_SOURCES = ["api.cu", "common.cuh", "gemv.cu", "gemvband.cu", "internal.h", "ptx.cuh", "sched.cuh",
                         "umma.cu", "waits.cuh"]


def kernel_sources_sha256():
    import hashlib
    csrc = os.path.join(ROOT, "dense_bit_weight_gb300", "csrc")
    h = hashlib.sha256()
    for f in DECODE_KERNEL_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "dbw_gemm.h"), "rb").read())
    return h.hexdigest()


def bytes_bf16(M, N, K):
    return 2 * (M * K + N * K + M * N)


def bytes_w4(M, N, K, g=128):
    return N * K // 2 + (N * K // g) * 3 + 2 * M * K + 2 * M * N


def flops(M, N, K):
    return 2 * M * N * K


def bytes_mx(M, N, K, fmt):
    el = 1 if fmt == "e4m3" else 0.5
    return int(el * (M * K + N * K) + (M * K + N * K) // 32 + 2 * M * N)


def mx_sweep(g, torch, reps=10):
    """Block-scaled GEMMs: TFLOP/s per shape (graph-timed, random codes drawn on
    the device; operands rotated over copies larger than L2) and the
    fraction of max(flops / P_fmt, bytes / BW), P_fmt = the measured bf16
    peak times the nominal format ratio."""
    hbm, tf, _, _ = peaks()
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    out = {}
    for fmt in ("e4m3", "e2m1"):
        p_fmt = tf * MX_PEAK_RATIO[fmt]
        rows, t_roof, t_meas = [], 0.0, 0.0
        for (M, N, K) in MX_SHAPES:
            w = K if fmt == "e4m3" else K // 2
            copies = max(1, min(6, int(np.ceil(3 * 126e6 / (N * w + M * w)))))
            def codes(r):   # E4M3: exponent fields 4..10 (no NaN); E2M1: any byte
                x = torch.randint(0, 256, (r, w), generator=gen, device=dev, dtype=torch.uint8)
                return (x & 0xB7) | 0x20 if fmt == "e4m3" else x
            ops = [(codes(M), torch.randint(124, 131, (M, K // 32), generator=gen, device=dev, dtype=torch.uint8),
                    codes(N), torch.randint(124, 131, (N, K // 32), generator=gen, device=dev, dtype=torch.uint8))
                   for _ in range(copies)]
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ms = graph_time_ms(torch, lambda i: g.gemm_mx(*ops[i % copies], fmt, C=C), reps)
            fl, by = flops(M, N, K), bytes_mx(M, N, K, fmt)
            tr = max(fl / (p_fmt * 1e12), by / (hbm * 1e9))
            t_roof += tr
            t_meas += ms * 1e-3
            rows.append([M, N, K, round(fl / (ms * 1e-3) / 1e12, 1), round(tr / (ms * 1e-3), 3)])
            del ops, C
        out[fmt] = {"unit": "[M, N, K, TFLOP/s, t_roof / t]", "peak_tflops": round(p_fmt, 1),
                    "peak_source": "measured bf16 x nominal ratio", "roofline_frac_aggregate": t_roof / t_meas,
                    "shapes": rows}
    return out


def roof_frac(M, N, K, ms, kind, hbm, tf):
    """t_roof / t_measured with t_roof = max(flops / P_tc, bytes / BW): the
    per-shape fraction of the roofline (a shape is graded on whichever side
    bounds it).  kind: "bf16" (bytes 2(MK + NK + MN)), "w4" (the W4A16 bytes)
    or "silu" (2N weight rows, C of N columns)."""
    if kind == "w4":
        fl, by = flops(M, N, K), bytes_w4(M, N, K)
    elif kind == "silu":
        fl, by = flops(M, 2 * N, K), 2 * (M * K + 2 * N * K + M * N)
    else:
        fl, by = flops(M, N, K), bytes_bf16(M, N, K)
    t_roof = max(fl / (tf * 1e12), by / (hbm * 1e9))
    return t_roof / (ms * 1e-3), t_roof


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # raw samples in the system temporary directory (the JSON line carries the summary)
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"dbw_clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- our arm

class Arm:
    """The GEMMs of one step, with device-resident operands."""

    def __init__(self, dev):
        import torch
        from dense_bit_weight_gb300 import gemm
        self.torch, self.g, self.dev = torch, gemm, dev
        self.stream = torch.cuda.current_stream(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(0)
        self.items = []
        for (M, N, K) in DECODE:
            A = (torch.randn((M, K), generator=gen, device=dev)).to(torch.bfloat16)
            B = (torch.randn((N, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            plan = gemm.gemm_bf16_plan(M, N, K)
            self.items.append(dict(M=M, N=N, K=K, A=A, B=B, C=C, plan=plan,
                                   name=self.kname(plan), bytes=bytes_bf16(M, N, K)))
        # GEMMs of one kernel family run back to back; timing events sit only
        # at family boundaries (an event between two kernels costs a launch gap)
        self.items.sort(key=lambda it: (it["name"], it["N"]))
        self.groups = []
        for i, it in enumerate(self.items):
            if not self.groups or self.groups[-1]["name"] != it["name"]:
                self.groups.append({"name": it["name"], "idx": []})
            self.groups[-1]["idx"].append(i)

    @staticmethod
    def kname(plan):
        # kernel family: the variant and its tile width (the template instance)
        return f"{plan['variant_name']}[tile {plan['tile_m']}x{plan['tile_n']}]"

    def call(self, it):
        rc = self.g.gemm_bf16_ptr(it["A"].data_ptr(), it["B"].data_ptr(), it["C"].data_ptr(),
                                  it["M"], it["N"], it["K"], it["K"], it["K"], it["N"],
                                  self.torch.cuda.current_stream().cuda_stream)
        if rc:
            raise self.g.GemmError(rc, "gemm_bf16")

    def step(self, events=None):
        cur = self.torch.cuda.current_stream()
        for gi, grp in enumerate(self.groups):
            if events is not None:
                events[gi][0].record(cur)
            for i in grp["idx"]:
                self.call(self.items[i])
            if events is not None:
                events[gi][1].record(cur)


def pack_e2e(torch, items, dev, pin=True):
    """One host buffer and one device buffer holding every GEMM's activations,
    and one pair holding every output, so an end-to-end step moves its inputs
    and its results with one copy each.  Returns (host_a, dev_a, host_c, dev_c,
    items) where the items' A and C are views of dev_a and dev_c (each view
    starts at a multiple of 8 elements: 16-byte aligned, as the library wants).
    The host activations hold the items' current values."""
    def offsets(sizes):
        out, o = [], 0
        for n in sizes:
            out.append(o)
            o += (n + 7) // 8 * 8
        return out, o
    a_off, a_tot = offsets([it["M"] * it["K"] for it in items])
    c_off, c_tot = offsets([it["M"] * it["N"] for it in items])
    host_a = torch.empty(a_tot, dtype=torch.bfloat16, pin_memory=pin)
    host_c = torch.empty(c_tot, dtype=torch.bfloat16, pin_memory=pin)
    dev_a = torch.empty(a_tot, dtype=torch.bfloat16, device=dev)
    dev_c = torch.empty(c_tot, dtype=torch.bfloat16, device=dev)
    packed = []
    for it, oa, oc in zip(items, a_off, c_off):
        M, N, K = it["M"], it["N"], it["K"]
        host_a[oa:oa + M * K].copy_(it["A"].reshape(-1))
        packed.append(dict(it, A=dev_a[oa:oa + M * K].view(M, K), C=dev_c[oc:oc + M * N].view(M, N)))
    return host_a, dev_a, host_c, dev_c, packed


def dist_init(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier_max(x, ws):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def graph_time_ms(torch, fn, reps):
    """Device time per call of fn, from one CUDA-graph replay of `reps` calls
    (captured after eager warm-up on the same stream, so the library's
    per-stream workspace exists before capture)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(reps):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def timed_sweep(g, torch, shapes, kind, reps=20):
    """Per-shape device time (ms per launch) for the extra sweeps."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    out = []
    for (M, N, K) in shapes:
        silu = kind.startswith("silu")
        NB = 2 * N if silu else N   # weight rows
        plan = (g.gemm_w4a16_plan(M, N, K, 128) if kind == "w4"
                else g.gemm_bf16_fused_plan(M, N, K, "silu_mul") if silu else g.gemm_bf16_plan(M, NB, K))
        if plan["variant"] == 1 and M > 64:
            continue            # no tensor-core plan for this shape
        # enough weight copies that consecutive launches miss L2
        wbytes = NB * K * 2 if kind != "w4" else N * K // 2
        copies = max(1, min(8, int(np.ceil(3 * 126e6 / wbytes))))
        A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        if kind == "w4":
            Bs = [(torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), generator=gen, device=dev, dtype=torch.int32),
                   (torch.rand((N, K // 128), generator=gen, device=dev) * 0.018 + 0.002).to(torch.bfloat16),
                   torch.randint(0, 16, (N, K // 128), generator=gen, device=dev, dtype=torch.uint8))
                  for _ in range(copies)]
            fn = lambda i: g.gemm_w4a16(A, *Bs[i % copies], 128, C)
            work = bytes_w4(M, N, K)
        elif silu:
            Bs = [(torch.randn((NB, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
                  for _ in range(copies)]
            fn = lambda i: g.gemm_bf16_fused(A, Bs[i % copies], C=C, epilogue="silu_mul")
            # algorithmic work: the 2N-row contraction; bytes read A and B, write C [M, N]
            work = flops(M, NB, K) if kind == "silu_prefill" else 2 * (M * K + NB * K + M * N)
        else:
            Bs = [(torch.randn((N, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
                  for _ in range(copies)]
            fn = lambda i: g.gemm_bf16(A, Bs[i % copies], C)
            work = flops(M, N, K) if kind == "prefill" else bytes_bf16(M, N, K)
        ms = graph_time_ms(torch, fn, reps)
        out.append({"M": M, "N": N, "K": K, "ms": ms, "work": work, "variant": plan["variant_name"]})
        del Bs, A, C
    return out


def grouped_sweep(g, torch, reps=20):
    """The grouped GEMM: useful TFLOP/s (2 * rows * N * K) and GB/s (A, the
    active experts' weights, C), graph-timed, weights rotated over copies."""
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(2)
    out = []
    for name, counts, N, K in GROUPED:
        G, M = len(counts), sum(counts)
        wbytes = G * N * K * 2
        copies = max(1, min(8, -(-3 * 130_000_000 // wbytes)))
        A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
        C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        Bs = [(torch.randn((G, N, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
              for _ in range(copies)]
        ends = torch.tensor(np.cumsum(counts), dtype=torch.int32, device=dev)
        ms = graph_time_ms(torch, lambda i: g.gemm_bf16_grouped(A, Bs[i % copies], ends, C=C), reps)
        active = sum(1 for c in counts if c)
        fl = 2 * M * N * K
        by = 2 * (M * K + active * N * K + M * N)
        out.append([name, M, N, K, round(fl / (ms * 1e-3) / 1e12, 1), round(by / (ms * 1e-3) / 1e9, 1)])
        del Bs, A, C
    return {"unit": "[name, rows, N, K, TFLOP/s, GB/s]", "shapes": out}


def cpu_oracle_sample(target_s=12.0):
    """Time the oracle on a fraction of every decode GEMM's output columns."""
    import oracle
    from dense_bit_weight_gb300 import synth
    cores = oracle.hardware_threads()
    # calibrate on a piece large enough that thread start-up does not count,
    # then size the sample for about target_s seconds
    A = synth.bf16_normal((8, 4096), 1.0, 0, synth.STREAM_A)
    B = synth.bf16_normal((4096, 4096), 4096 ** -0.5, 0, synth.STREAM_B)
    t = time.perf_counter()
    oracle.gemm_bf16(A, B)
    per_mac = (time.perf_counter() - t) / (8 * 4096 * 4096)
    total_macs = sum(M * N * K for (M, N, K) in DECODE)
    frac = min(1.0, target_s / max(per_mac * total_macs, 1e-9))
    work, secs = 0, 0.0
    for (M, N, K) in DECODE:
        n = max(8, int(N * frac))
        A = synth.bf16_normal((M, K), 1.0, 0, synth.STREAM_A)
        B = synth.bf16_normal((n, K), K ** -0.5, 0, synth.STREAM_B)
        t = time.perf_counter()
        oracle.gemm_bf16(A, B)
        secs += time.perf_counter() - t
        work += bytes_bf16(M, n, K)
    return {"value": work / secs / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"every decode GEMM on the first {frac:.2%} of its weight rows "
                      f"({work / 1e6:.1f} MB algorithmic, {secs:.1f} s)"}, secs


def cpu_oracle_configs(seconds_each=4.0):
    """The oracle on a bounded sample of each other config (down projection,
    prefill sweep, W4A16 decode): every shape of the config on its first rows
    of C (rows of A for prefill, weight rows for the decode-like configs),
    sized for about `seconds_each` seconds per config.  Rates are of the
    sampled work: GFLOP/s (2 * MACs) and algorithmic GB/s of the sampled
    operands."""
    import oracle
    from dense_bit_weight_gb300 import synth
    # calibration: MACs per second of each oracle routine on this host
    A = synth.bf16_normal((8, 4096), 1.0, 0, synth.STREAM_A)
    B = synth.bf16_normal((2048, 4096), 4096 ** -0.5, 0, synth.STREAM_B)
    t = time.perf_counter()
    oracle.gemm_bf16(A, B)
    bf16_mac_s = 8 * 2048 * 4096 / (time.perf_counter() - t)
    Bq, S, Z = synth.w4a16_operands(2048, 4096, 128, 0)
    t = time.perf_counter()
    oracle.gemm_w4a16(A, Bq, S, Z, 128)
    w4_mac_s = 8 * 2048 * 4096 / (time.perf_counter() - t)
    out = {}
    for name, shapes, kind in (("down", DOWN, "bf16"), ("prefill", PREFILL, "bf16"), ("w4a16", W4, "w4")):
        rate = w4_mac_s if kind == "w4" else bf16_mac_s
        total = sum(M * N * K for (M, N, K) in shapes)
        frac = min(1.0, seconds_each * rate / total)
        macs, by, secs = 0, 0, 0.0
        for (M, N, K) in shapes:
            if name == "prefill":       # the first m token rows against all weights
                m, n = max(1, int(M * frac)), N
            else:                       # all tokens against the first n weight rows
                m, n = M, max(8, int(N * frac) // 8 * 8)
            A = synth.bf16_normal((m, K), 1.0, 0, synth.STREAM_A)
            if kind == "w4":
                Bq, S, Z = synth.w4a16_operands(n, K, 128, 0)
                t = time.perf_counter()
                oracle.gemm_w4a16(A, Bq, S, Z, 128)
                by += bytes_w4(m, n, K)
            else:
                B = synth.bf16_normal((n, K), K ** -0.5, 0, synth.STREAM_B)
                t = time.perf_counter()
                oracle.gemm_bf16(A, B)
                by += bytes_bf16(m, n, K)
            secs += time.perf_counter() - t
            macs += m * n * K
        out[name] = {"GFLOP/s": round(2 * macs / secs / 1e9, 3), "GB/s": round(by / secs / 1e9, 4),
                     "sample": f"every shape on {'the first' if name == 'prefill' else 'all tokens x the first'} "
                               f"{frac:.3%} of its {'token rows' if name == 'prefill' else 'weight rows'} "
                               f"({2 * macs / 1e9:.1f} GFLOP, {secs:.1f} s)"}
    return out


def run_ours(args):
    import torch
    ws, rank, local = dist_init(args)
    torch.cuda.synchronize()
    arm = Arm(torch.device("cuda", torch.cuda.current_device()))
    g = arm.g
    n_items = len(arm.items)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):          # warm-up (also creates the stream's workspace)
        for _ in range(args.warmup):
            arm.step()
    torch.cuda.synchronize()

    # The timed region replays a CUDA graph of S steps (plus one of K % S steps)
    # so exactly K steps run back to back with no host launch gaps and no
    # timing events between GEMMs.  A second graph of the same S steps, with a
    # pair of events around each kernel family's GEMMs, is replayed afterwards
    # over K steps for the per-kernel durations (an event between two kernels
    # costs a launch gap, so it is kept out of the headline region).
    S = max(1, min(args.steps, args.graph_steps))
    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)
        mk()
    except TypeError:
        mk = None
    n_groups = len(arm.groups)

    def capture(nsteps, with_events):
        evs = [[(mk(), mk()) for _ in range(n_groups)] for _ in range(nsteps)] if (with_events and mk) else None
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for k in range(nsteps):
                arm.step(evs[k] if evs else None)
        return gr, evs

    graph, _ = capture(S, False)
    rest = args.steps % S
    graph_rest, _ = capture(rest, False) if rest else (None, None)
    graph_ev, events = capture(S, True)
    with torch.cuda.stream(stream):
        graph.replay()
        graph_ev.replay()
    torch.cuda.synchronize()

    def replay_steps(g_main, g_rest):
        for _ in range(args.steps // S):
            g_main.replay()
        if g_rest is not None:
            g_rest.replay()

    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    # keep the GPU under the same load around the timed region so the clock
    # samples (every 200 ms) see the loaded state
    t_end = time.time() + args.preroll
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            graph.replay()
            torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        replay_steps(graph, graph_rest)
        t1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    # the per-kernel replays (same load, inside the clock window)
    group_ms = [0.0] * n_groups
    nsteps = 0
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.steps // S)):
            graph_ev.replay()
            torch.cuda.synchronize()
            if events is not None:
                for k in range(S):
                    for gi in range(n_groups):
                        group_ms[gi] += events[k][gi][0].elapsed_time(events[k][gi][1])
            nsteps += S
    t_end = time.time() + args.preroll
    with torch.cuda.stream(stream):
        while time.time() < t_end:
            graph.replay()
            torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = barrier_max(t0.elapsed_time(t1), ws)
    step_bytes = sum(it["bytes"] for it in arm.items)
    value = ws * step_bytes * args.steps / (ms_total * 1e-3) / 1e9

    per = {}
    if events is None:
        # no external events in this torch: time each family alone in a graph of S steps
        nsteps = S
        for gi, grp in enumerate(arm.groups):
            calls = [arm.items[i] for i in grp["idx"]]
            group_ms[gi] = graph_time_ms(torch, lambda _k, calls=calls: [arm.call(c) for c in calls], S) * S
    for gi, grp in enumerate(arm.groups):
        its = [arm.items[i] for i in grp["idx"]]
        per[grp["name"]] = {"ms": group_ms[gi], "bytes": sum(it["bytes"] for it in its) * nsteps,
                            "launches": sum(it["plan"]["kernels"] for it in its) * nsteps,
                            "shapes": [[it["M"], it["N"], it["K"]] for it in its],
                            "traffic": [TRAFFIC_BYTES.get((it["M"], it["N"], it["K"])) for it in its]}
    dom_name = max(per, key=lambda k: per[k]["ms"])
    dom = per[dom_name]
    hbm, tf, tf_sus, src = peaks()
    achieved = dom["bytes"] / (dom["ms"] * 1e-3) / 1e9
    traffic = None
    if kernel_sources_sha256() == TRAFFIC_SOURCES_SHA256 and None not in dom["traffic"]:
        traffic = round(sum(dom["traffic"]) / len(dom["traffic"]))     # bytes per launch, family average
    gpu_launches = sum(it["plan"]["kernels"] for it in arm.items) * args.steps

    # end to end through the public call, host buffers, copies inside the
    # timing: every step copies all its activations in (one pinned buffer) and
    # all its outputs out (one pinned buffer)
    host_a, dev_a, host_c, dev_c, e2e_items = pack_e2e(torch, arm.items, arm.dev)
    e2e_steps = max(1, min(args.steps, 10))

    def e2e_step():
        dev_a.copy_(host_a, non_blocking=True)
        for it in e2e_items:
            arm.call(it)
        host_c.copy_(dev_c, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_steps):
        e2e_step()
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = barrier_max(e0.elapsed_time(e1), ws)
    h2d = host_a.numel() * host_a.element_size()    # bytes of the two copies of a step
    d2h = host_c.numel() * host_c.element_size()
    e2e = {"value": ws * step_bytes * e2e_steps / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    sweeps = None
    if rank == 0 and not args.no_sweeps:
        sweeps = {}

        def graded(rs, kind):
            # per shape: [M, N, K, rate, variant, t_roof / t_measured]; aggregate: sum t_roof / sum t
            shapes, t_roof, t_meas = [], 0.0, 0.0
            for r in rs:
                f, tr = roof_frac(r["M"], r["N"], r["K"], r["ms"], kind, hbm, tf)
                t_roof += tr
                t_meas += r["ms"] * 1e-3
                shapes.append(round(f, 3))
            return shapes, (t_roof / t_meas if t_meas else None)
        pre = timed_sweep(g, torch, PREFILL, "prefill") if not args.quick else []
        if pre:
            tot_f = sum(r["work"] for r in pre)
            tot_ms = sum(r["ms"] for r in pre)
            sweeps["prefill"] = {"unit": "TFLOP/s", "aggregate": tot_f / (tot_ms * 1e-3) / 1e12,
                                 "frac_of_peak": tot_f / (tot_ms * 1e-3) / 1e12 / tf,
                                 "shapes": [[r["M"], r["N"], r["K"], round(r["work"] / (r["ms"] * 1e-3) / 1e12, 1),
                                             r["variant"]] for r in pre]}
            fr, agg = graded(pre, "bf16")
            sweeps["prefill"]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        for key, shapes, kind in (("down", DOWN, "bf16"), ("w4a16", W4, "w4")):
            rs = timed_sweep(g, torch, shapes, kind)
            tot_b = sum(r["work"] for r in rs)
            tot_ms = sum(r["ms"] for r in rs)
            sweeps[key] = {"unit": "GB/s", "aggregate": tot_b / (tot_ms * 1e-3) / 1e9,
                           "frac_of_peak": tot_b / (tot_ms * 1e-3) / 1e9 / hbm,
                           "shapes": [[r["M"], r["N"], r["K"], round(r["work"] / (r["ms"] * 1e-3) / 1e9, 1),
                                       r["variant"]] for r in rs]}
            fr, agg = graded(rs, kind)
            sweeps[key]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        rs = timed_sweep(g, torch, W4_PREFILL, "w4", reps=10) if not args.quick else []
        if rs:
            tot_f = sum(flops(r["M"], r["N"], r["K"]) for r in rs)
            tot_ms = sum(r["ms"] for r in rs)
            sweeps["w4a16_prefill"] = {
                "unit": "TFLOP/s", "aggregate": tot_f / (tot_ms * 1e-3) / 1e12, "frac_of_peak": tot_f / (tot_ms * 1e-3) / 1e12 / tf,
                "shapes": [[r["M"], r["N"], r["K"], round(flops(r["M"], r["N"], r["K"]) / (r["ms"] * 1e-3) / 1e12, 1),
                            r["variant"]] for r in rs]}
            fr, agg = graded(rs, "w4")
            sweeps["w4a16_prefill"]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        # the fused gate/up projection with the SiLU-mul epilogue
        rs = timed_sweep(g, torch, GATE_UP_DECODE, "silu")
        tot_b, tot_ms = sum(r["work"] for r in rs), sum(r["ms"] for r in rs)
        sweeps["gate_up_silu_decode"] = {
            "unit": "GB/s", "aggregate": tot_b / (tot_ms * 1e-3) / 1e9, "frac_of_peak": tot_b / (tot_ms * 1e-3) / 1e9 / hbm,
            "shapes": [[r["M"], r["N"], r["K"], round(r["work"] / (r["ms"] * 1e-3) / 1e9, 1), r["variant"]] for r in rs]}
        fr, agg = graded(rs, "silu")
        sweeps["gate_up_silu_decode"]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        rs = timed_sweep(g, torch, GATE_UP_PREFILL, "silu_prefill") if not args.quick else []
        if rs:
            tot_f, tot_ms = sum(r["work"] for r in rs), sum(r["ms"] for r in rs)
            sweeps["gate_up_silu_prefill"] = {
                "unit": "TFLOP/s", "aggregate": tot_f / (tot_ms * 1e-3) / 1e12, "frac_of_peak": tot_f / (tot_ms * 1e-3) / 1e12 / tf,
                "shapes": [[r["M"], r["N"], r["K"], round(r["work"] / (r["ms"] * 1e-3) / 1e12, 1), r["variant"]]
                           for r in rs]}
            fr, agg = graded(rs, "silu")
            sweeps["gate_up_silu_prefill"]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        sweeps["grouped"] = grouped_sweep(g, torch)
        if not args.quick:
            sweeps["mx"] = mx_sweep(g, torch)
        # each decode shape alone, graph-timed back to back (no events between launches)
        dec = timed_sweep(g, torch, DECODE, "bf16")
        sweeps["decode_per_shape"] = {"unit": "GB/s", "shapes": [
            [r["M"], r["N"], r["K"], round(r["work"] / (r["ms"] * 1e-3) / 1e9, 1), r["variant"]]
            for r in dec]}
        fr, agg = graded(dec, "bf16")
        sweeps["decode_per_shape"]["roofline_frac"] = {"per_shape": fr, "aggregate": agg}
        sweeps["roofline_peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tf, "source": src,
                                    "t_roof": "max(2MNK / bf16_tflops, algorithmic bytes / hbm_gbs)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu, _ = cpu_oracle_sample(args.cpu_seconds)
        if not args.no_sweeps:
            cpu["other_configs"] = cpu_oracle_configs()

    err = g.gemm_last_device_error()
    if err:
        raise RuntimeError(f"device error word set: {g.gemm_status_string(err)}")
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_total / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "gemms_per_step": n_items,
                       "timing": f"CUDA graph of {S} steps replayed with no events between GEMMs; "
                                 "per-kernel durations from a second replay with events around each "
                                 "kernel family's GEMMs",
                       "l2": "inputs larger than L2: each GEMM has its own weight copy, "
                             f"{step_bytes / 1e9:.2f} GB streamed per step",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "peak_source": src, "traffic": traffic,
                         "algorithmic_bytes_per_launch": round(dom["bytes"] / dom["launches"])},
            "e2e": {k: (round(v, 2) if isinstance(v, float) else v) for k, v in e2e.items()},
            "cpu_baseline": cpu,
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "per_kernel": {k: {"launches": v["launches"], "ms": round(v["ms"], 4),
                               "GB/s": round(v["bytes"] / (v["ms"] * 1e-3) / 1e9, 1),
                               "shapes": v["shapes"]}
                           for k, v in per.items()},
            "sweeps": sweeps,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle (fp64 CPU definition) on the host cores, rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from dense_bit_weight_gb300 import synth
    cores = oracle.hardware_threads()
    # each step: every decode GEMM on a slice of its weight rows, about 1 s of CPU work
    A = synth.bf16_normal((8, 4096), 1.0, 0, synth.STREAM_A)
    Bc = synth.bf16_normal((4096, 4096), 4096 ** -0.5, 0, synth.STREAM_B)
    t = time.perf_counter()
    oracle.gemm_bf16(A, Bc)
    per_mac = (time.perf_counter() - t) / (8 * 4096 * 4096)
    total = sum(M * N * K for (M, N, K) in DECODE)
    frac = min(1.0, args.ref_step_seconds / max(per_mac * total, 1e-9))
    ops = []
    for (M, N, K) in DECODE:
        n = max(8, int(N * frac))
        ops.append((synth.bf16_normal((M, K), 1.0, 0, synth.STREAM_A),
                    synth.bf16_normal((n, K), K ** -0.5, 0, synth.STREAM_B), bytes_bf16(M, n, K)))
    step_bytes = sum(o[2] for o in ops)

    def step():
        for a, b, _ in ops:
            oracle.gemm_bf16(a, b)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t
    value = step_bytes * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemms_per_step": len(ops),
                   "l2": "host oracle; no device caches involved",
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: every decode GEMM on the first {frac:.2%} of its "
                                   f"weight rows ({step_bytes / 1e6:.1f} MB algorithmic)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--graph-steps", type=int, default=50,
                    help="steps per captured CUDA graph (the timed region replays it)")
    ap.add_argument("--preroll", type=float, default=0.6,
                    help="seconds of untimed load before and after the timed region (clock sampling)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweeps", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the prefill sweep")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=1.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
