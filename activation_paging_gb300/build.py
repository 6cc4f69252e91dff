"""Build ``libap.so`` (the CUDA library behind ``include/ap.h``) in-tree.

Each ``csrc/*.cu`` file is compiled for sm_103a in parallel, then linked into
a shared library next to this file.  The CUDA runtime is linked statically, so
the library needs only the driver at run time.

    python -m activation_paging_gb300.build          # build if stale
    AP_PTXAS_VERBOSE=1 python -m activation_paging_gb300.build --force
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libap.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["common.cu", "route.cu", "dispatch.cu", "combine.cu", "stash.cu", "noalloc.cu", "arena.cu"]
# bench-only synthetic compute (whole-SM busy blocks for the overlap measurement), not part of libap.so
BENCH_SOURCES = ["bench/busy.cu", "bench/green.cu"]
BENCH_LIB = os.path.join(HERE, "libap_bench.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if os.path.isfile(os.path.join(CSRC, f))]
    files += [os.path.join(CSRC, s) for s in BENCH_SOURCES]
    files.append(os.path.join(INCLUDE, "ap.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(BENCH_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(BENCH_LIB))
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE]
    if os.environ.get("AP_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    bench_objs = []
    for src in _sources() + BENCH_SOURCES:
        obj = os.path.join(BUILD, src.replace("/", "_").replace(".cu", ".o"))
        (bench_objs if src in BENCH_SOURCES else objs).append(obj)
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(src)
            sys.stderr.write(text)
        elif text.strip() and (verbose or os.environ.get("AP_PTXAS_VERBOSE")):
            sys.stdout.write(text)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    for lib, lib_objs in ((LIB, objs), (BENCH_LIB, bench_objs)):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *lib_objs], check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
