"""Builds libmuon.so (the Muon step), libmuon_debug.so (the same with the device
range checks of -DMUON_DEBUG) and libmuonsynth.so (seeded input fill) in-tree.

nvcc compiles each translation unit for sm_103a in parallel, then links a
shared library next to the sources.  No CMake, no torch extension machinery.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]

LIBMUON = os.path.join(PKG, "libmuon.so")
LIBMUON_DEBUG = os.path.join(PKG, "libmuon_debug.so")
LIBSYNTH = os.path.join(ROOT, "synth", "libmuonsynth.so")

MUON_SOURCES = ["runtime.cu", "elementwise.cu", "ns_gemm.cu", "ns_small.cu", "ns_gram.cu", "noalloc.cu",
                "schedule.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r


def _newer(target: str, sources) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def build(verbose: bool = False, force: bool = False) -> None:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "muon.h"))
    os.makedirs(os.path.join(BUILD, "debug"), exist_ok=True)
    jobs = []
    objs, dobjs = [], []
    for src in MUON_SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        d = os.path.join(BUILD, "debug", src.replace(".cu", ".o"))
        objs.append(o)
        dobjs.append(d)
        if force or not _newer(o, [s] + headers):
            jobs.append([nvcc, *ARCH, *COMMON, "-c", s, "-o", o])
        if force or not _newer(d, [s] + headers):
            jobs.append([nvcc, *ARCH, *COMMON, "-DMUON_DEBUG", "-c", s, "-o", d])
    synth_src = os.path.join(ROOT, "synth", "csrc", "synth.cu")
    synth_obj = os.path.join(BUILD, "synth.o")
    if force or not _newer(synth_obj, [synth_src]):
        # no multiply-add contraction: the fill must match the numpy generator bit for bit
        jobs.append([nvcc, *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false",
                     "-c", synth_src, "-o", synth_obj])
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for r in ex.map(_run, jobs):
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr, file=sys.stderr)
    if force or not _newer(LIBMUON, objs):
        _run([nvcc, *ARCH, "-shared", "-o", LIBMUON, *objs])
    if force or not _newer(LIBMUON_DEBUG, dobjs):
        _run([nvcc, *ARCH, "-shared", "-o", LIBMUON_DEBUG, *dobjs])
    if force or not _newer(LIBSYNTH, [synth_obj]):
        _run([nvcc, *ARCH, "-shared", "-o", LIBSYNTH, synth_obj])


if __name__ == "__main__":
    build(verbose=True, force="--force" in sys.argv)
    print(LIBMUON)
    print(LIBMUON_DEBUG)
    print(LIBSYNTH)
