"""Run one GEMM shape repeatedly on the GPU (for profiling and quick timing).

    python run_case.py --M 1 --N 24576 --K 4096 \
        [--kind bf16|w4a16|silu_mul|grouped|mxfp8|mxfp4] [--variant auto|gemv|skinny|prefill]
        [--groups G] [--reps 4] [--copies 0]

--kind silu_mul runs the fused gate/up projection (C [M,N], weights 2N rows);
--kind grouped runs the grouped GEMM with M tokens split evenly over G experts;
--kind mxfp8 / mxfp4 the block-scaled GEMM on random E4M3 / packed E2M1 codes
with random E8M0 scales (one per 32 along K).

Weights are drawn on the device with torch's seeded generator; `--copies`
weight copies (0 = enough to exceed three L2 sizes) are used round robin so
every launch streams its weights from HBM.  Prints the plan and the mean
device time per launch of a CUDA-graph replay.  Meant to be run under
`ncu -k regex:<kernel> -s <skip> -c <count>`.
"""
from __future__ import annotations

import argparse
import json
import math


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--M", type=int, required=True)
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, required=True)
    ap.add_argument("--kind", choices=["bf16", "w4a16", "silu_mul", "grouped", "mxfp8", "mxfp4"], default="bf16")
    ap.add_argument("--groups", type=int, default=8)
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--group", type=int, default=128)
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--copies", type=int, default=0)
    ap.add_argument("--no-graph", action="store_true", help="eager launches only (for ncu)")
    a = ap.parse_args(argv)

    import torch
    from dense_bit_weight_gb300 import gemm as g

    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    M, N, K = a.M, a.N, a.K
    NB = 2 * N if a.kind == "silu_mul" else a.groups * N if a.kind == "grouped" else N   # weight rows
    wbytes = (N * K // 2 if a.kind in ("w4a16", "mxfp4") else N * K if a.kind == "mxfp8" else NB * K * 2)
    copies = a.copies or max(1, min(16, math.ceil(3 * 130e6 / wbytes)))
    A = torch.randn((M, K), generator=gen, device=dev).to(torch.bfloat16)
    C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if a.kind == "silu_mul":
        Bs = [(torch.randn((NB, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
              for _ in range(copies)]
        plan = g.gemm_bf16_plan(M, NB, K, a.variant)
        fn = lambda i: g.gemm_bf16_fused(A, Bs[i % copies], C=C, epilogue="silu_mul", variant=a.variant)
        work = {"GB": 2 * (M * K + NB * K + M * N) / 1e9, "TFLOP": 2 * M * NB * K / 1e12}
    elif a.kind == "grouped":
        Bs = [(torch.randn((a.groups, N, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
              for _ in range(copies)]
        ends = torch.tensor([M * (e + 1) // a.groups for e in range(a.groups)], dtype=torch.int32, device=dev)
        plan = {"variant_name": "prefill (grouped)", "groups": a.groups}
        fn = lambda i: g.gemm_bf16_grouped(A, Bs[i % copies], ends, C=C)
        work = {"GB": 2 * (M * K + NB * K + M * N) / 1e9, "TFLOP": 2 * M * N * K / 1e12}
    elif a.kind in ("mxfp8", "mxfp4"):
        fmt = "e4m3" if a.kind == "mxfp8" else "e2m1"
        kb = K if fmt == "e4m3" else K // 2   # bytes per row
        rnd = lambda r, c: torch.randint(0, 256, (r, c), generator=gen, device=dev, dtype=torch.uint8)
        codes = lambda r, c: (rnd(r, c) & 0x77) if fmt == "e4m3" else rnd(r, c)   # E4M3: no NaN codes
        scales = lambda r: torch.randint(124, 131, (r, K // 32), generator=gen, device=dev, dtype=torch.uint8)
        A = codes(M, kb)
        SA = scales(M)
        Bs = [(codes(N, kb), scales(N)) for _ in range(copies)]
        plan = g.gemm_mx_plan(M, N, K, fmt)
        fn = lambda i: g.gemm_mx(A, SA, Bs[i % copies][0], Bs[i % copies][1], fmt, C)
        work = {"GB": ((M + N) * kb + (M + N) * K // 32 + 2 * M * N) / 1e9, "TFLOP": 2 * M * N * K / 1e12}
    elif a.kind == "bf16":
        Bs = [(torch.randn((N, K), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
              for _ in range(copies)]
        plan = g.gemm_bf16_plan(M, N, K, a.variant)
        fn = lambda i: g.gemm_bf16(A, Bs[i % copies], C, variant=a.variant)
        work = {"GB": 2 * (M * K + N * K + M * N) / 1e9, "TFLOP": 2 * M * N * K / 1e12}
    else:
        G = K // a.group
        Bs = [(torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), generator=gen, device=dev, dtype=torch.int32),
               (torch.rand((N, G), generator=gen, device=dev) * 0.018 + 0.002).to(torch.bfloat16),
               torch.randint(0, 16, (N, G), generator=gen, device=dev, dtype=torch.uint8))
              for _ in range(copies)]
        plan = g.gemm_w4a16_plan(M, N, K, a.group, a.variant)
        fn = lambda i: g.gemm_w4a16(A, *Bs[i % copies], a.group, C, variant=a.variant)
        work = {"GB": (N * K // 2 + 3 * N * K // a.group + 2 * M * K + 2 * M * N) / 1e9,
                "TFLOP": 2 * M * N * K / 1e12}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(a.reps):
            fn(i)
    torch.cuda.synchronize()
    ms = None
    if not a.no_graph:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            for i in range(a.reps):
                fn(i)
        gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            gr.replay()
            e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / a.reps
    err = g.gemm_last_device_error()
    out = {"M": M, "N": N, "K": K, "kind": a.kind, "plan": plan, "copies": copies,
           "ms_per_launch": ms, "device_error": err}
    if ms:
        out["GB/s"] = work["GB"] / (ms * 1e-3)
        out["TFLOP/s"] = work["TFLOP"] / (ms * 1e-3)
    print(json.dumps(out))
    return 0 if err == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
