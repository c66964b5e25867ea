"""Build libdspark.so in-tree (``dspark_draft_sampling_gb300/_build/``) with nvcc for sm_103a.

Usage: ``python -m dspark_draft_sampling_gb300.build [--verbose-ptxas]``.
Translation units compile in parallel, then link against the shared CUDA runtime.
A second, small library, libdspark_bench.so, holds the measurement kernels bench.py uses
for the L2 / DRAM read bandwidth and the event-timing floor (``include/dspark_bench.h``).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
SRC_DIR = os.path.join(PKG_DIR, "csrc")
INCLUDE_DIR = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libdspark.so"
SOURCES = ["common.cu", "markov.cu", "markov_tc.cu", "markov_cluster.cu", "probe.cu", "ws_matvec.cu", "draft_plan.cu", "gated_plan.cu", "ws_q8.cu", "host_api.cu"]
BENCH_LIB_NAME = "libdspark_bench.so"
BENCH_SOURCES = ["bench_kernels.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libdspark")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def lib_file() -> str:
    return os.path.join(BUILD_DIR, LIB_NAME)


def bench_lib_file() -> str:
    return os.path.join(BUILD_DIR, BENCH_LIB_NAME)


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    headers = [os.path.join(SRC_DIR, h) for h in ("common.cuh", "markov.cuh", "tc.cuh")]
    headers += [os.path.join(INCLUDE_DIR, h) for h in ("dspark.h", "dspark_bench.h")]
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE_DIR, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]
    targets = [(lib_file(), SOURCES), (bench_lib_file(), BENCH_SOURCES)]
    objs_of, procs = {}, []
    for lib, srcs in targets:
        objs_of[lib] = []
        for src in srcs:
            s = os.path.join(SRC_DIR, src)
            o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
            objs_of[lib].append(o)
            if force or verbose_ptxas or _stale(o, [s] + headers):
                procs.append((src, subprocess.Popen([nvcc, *common, "-c", s, "-o", o],
                                                    stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif text.strip() and verbose_ptxas:
            sys.stdout.write(f"--- {src}\n{text}")
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    for lib, objs in objs_of.items():
        if force or _stale(lib, objs):
            tmp = lib + f".{os.getpid()}.tmp"
            cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "shared",
                   "-Xlinker", f"-rpath,{_cuda_lib_dir(nvcc)}"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, lib)
    return lib_file()


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(path)
