"""Build libhq.so (the CUDA library behind include/hq.h) in-tree, for sm_103a only.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared object with the CUDA runtime linked statically.  No fast-math: the
quantizers take integer decisions with IEEE fp32 division.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhq.so")
# (source, extra defines, object name): the kernel file is compiled in five parts
# (Q8_0, Q4_0, int8 and helpers, MoE, Q4_K)
SOURCES = [("hq_api.cu", [], "hq_api.o"), ("hq_quant.cu", [], "hq_quant.o")] + [
    ("hq_kernels.cu", [f"-DHQ_PART={i}"], f"hq_kernels_{i}.o") for i in range(5)]
HEADERS = ["hq_device.cuh", "hq_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-DNDEBUG"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    header_deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(HERE, "..", "include", "hq.h")]
    flags = NVCC_FLAGS + (extra_flags or [])
    jobs = []
    objs = []
    for src, defs, obj in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, obj)
        objs.append(o)
        if force or _stale(o, [s] + header_deps + [__file__]):
            jobs.append([nvcc, *ARCH, *flags, *defs, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or _stale(LIB, objs):
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", LIB + ".tmp", *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(LIB + ".tmp", LIB)
    return LIB


def kernel_resources(out_dir: str) -> dict:
    """Compile the kernel translation units (not linked, not installed) into
    `out_dir` with `ptxas -v` and return {mangled kernel name: (registers per
    thread, spill store bytes, spill load bytes)}."""
    import re
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    jobs = [[nvcc, *ARCH, *NVCC_FLAGS, "-Xptxas", "-v", *defs, "-c", os.path.join(CSRC, src),
             "-o", os.path.join(out_dir, obj)]
            for src, defs, obj in SOURCES if src == "hq_kernels.cu"]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    res, name, spill = {}, None, (0, 0)
    for r in results:
        if r.returncode != 0:
            raise RuntimeError("nvcc failed: " + r.stderr[-2000:])
        for ln in r.stderr.splitlines():
            m = re.search(r"Compiling entry function '([^']+)'", ln)
            if m:
                name = m.group(1)
                continue
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", ln)
            if m:
                spill = (int(m.group(1)), int(m.group(2)))
                continue
            m = re.search(r"Used (\d+) registers", ln)
            if m and name:
                res[name] = (int(m.group(1)), *spill)
                name, spill = None, (0, 0)
    return res


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))
