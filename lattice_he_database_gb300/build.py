"""Build the CUDA library libpir.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into a shared
library with the CUDA runtime linked statically.  No cmake, no torch
extension machinery: the library exposes a plain C ABI (include/pir.h).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpir.so")
SOURCES = ["ctx.cu", "ntt.cu", "encode.cu", "rowsel.cu", "rowsel_tc.cu", "scalar.cu", "server.cu", "coltor.cu", "expand.cu"]
HEADERS = ["common.cuh", "ntt_core.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def compile_units(sources, src_dir, out_lib, extra=(), force=False, verbose=False):
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(src_dir, s) for s in sources]
    deps = srcs + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "pir.h")]
    if not force and os.path.exists(out_lib) and os.path.getmtime(out_lib) >= _newest(deps):
        return out_lib
    procs, objs = [], []
    tag = os.path.basename(out_lib).replace(".so", "")
    for s in srcs:
        obj = os.path.join(BUILD, "%s_%s.o" % (tag, os.path.basename(s).replace(".cu", "")))
        objs.append(obj)
        cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", s, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(s)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = out_lib + ".tmp%d" % os.getpid()
    subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, out_lib)
    return out_lib


def build(force: bool = False, verbose: bool = False) -> str:
    return compile_units(SOURCES, CSRC, LIB, force=force, verbose=verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
