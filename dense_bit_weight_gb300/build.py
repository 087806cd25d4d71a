"""Build libdbw_gemm.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3 -Xptxas -v`` and the
objects are linked into ``dense_bit_weight_gb300/_build/libdbw_gemm.so``
(static CUDA runtime, no torch).  The build fails if ptxas reports any spill
or local-memory use in a kernel (the spill gate); ptxas' per-kernel report
is kept in ``_build/ptxas.log``.  Rebuilds are skipped when the sources and
flags are unchanged.
"""
from __future__ import annotations

import hashlib
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libdbw_gemm.so")
SOURCES = ["api.cu", "gemv.cu", "gemvband.cu", "w4band.cu", "umma.cu", "umma2.cu", "w4mma.cu", "w4frag.cu", "w4gemv.cu", "w4tc.cu", "mxgemm.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-Xptxas", "-v", "--expt-relaxed-constexpr", f"-I{INCLUDE}"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdbw_gemm.so")


def _digest() -> str:
    h = hashlib.sha256()
    files = sorted(os.listdir(CSRC)) + ["../../include/dbw_gemm.h"]
    for f in files:
        p = os.path.normpath(os.path.join(CSRC, f))
        if os.path.isfile(p):
            h.update(f.encode())
            h.update(open(p, "rb").read())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


_SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
_STACK = re.compile(r"(\d+) bytes stack frame")


def _spill_gate(log: str) -> list[str]:
    bad = []
    func = None
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'|Function properties for (\S+)", line)
        if m:
            func = m.group(1) or m.group(2)
        s = _SPILL.search(line)
        if s and (int(s.group(1)) or int(s.group(2))):
            bad.append(f"{func}: {line.strip()}")
    return bad


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    stamp = os.path.join(OUT, "stamp")
    dig = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == dig:
        return LIB
    nvcc = _nvcc()
    procs = []
    for src in SOURCES:
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                  stderr=subprocess.STDOUT, text=True)))
    logs, objs, failed = [], [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        logs.append(f"==== {src}\n{out}")
        objs.append(obj)
        if p.returncode != 0:
            failed.append(src)
    log = "\n".join(logs)
    with open(os.path.join(OUT, "ptxas.log"), "w") as f:
        f.write(log)
    if failed:
        sys.stderr.write(log)
        raise RuntimeError(f"nvcc failed for {failed}")
    bad = _spill_gate(log)
    if bad:
        sys.stderr.write("\n".join(bad) + "\n")
        raise RuntimeError("spill gate: a kernel spills registers or uses local memory")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lrt"],
                   check=True)
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(dig)
    if verbose:
        print(log)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
