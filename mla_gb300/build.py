"""Build step: compile the CUDA sources for sm_103a into in-tree shared libraries.

  mla_gb300/libmla.so          the MLA library (csrc/*.cu), C ABI in include/mla.h
  synth/libmlasynth.so         the seeded input generator's GPU copy
  tests/hooks/libmla_debug.so  test-only: the library's objects plus the test
                               hooks of tests/hooks/mla_debug.h

Translation units compile in parallel; only nvcc and the CUDA runtime
(statically linked) are needed, so the same step runs on the x86 dev host
(cross-compiling) and on the aarch64 GPU host.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mla_gb300")
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmla.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "synth.cu")
SYNTH_LIB = os.path.join(ROOT, "synth", "libmlasynth.so")
HOOKS_SRC = os.path.join(ROOT, "tests", "hooks", "mla_debug_hooks.cu")
HOOKS_LIB = os.path.join(ROOT, "tests", "hooks", "libmla_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    return r.stdout


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_verbose: bool = False) -> None:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers += [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    jobs = []
    objs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if _stale(obj, [src] + headers) or ptxas_verbose:
            extra = ["-Xptxas", "-v"] if ptxas_verbose else []
            jobs.append([cc, *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj])
    hooks_obj = os.path.join(BUILD, "mla_debug_hooks.o")
    hooks_deps = [HOOKS_SRC, os.path.join(ROOT, "tests", "hooks", "mla_debug.h")] + headers
    if os.path.exists(HOOKS_SRC) and (_stale(hooks_obj, hooks_deps) or ptxas_verbose):
        jobs.append([cc, *ARCH, *CFLAGS, "-c", HOOKS_SRC, "-o", hooks_obj])
    synth_job = None
    if _stale(SYNTH_LIB, [SYNTH_SRC]):
        synth_job = [cc, *ARCH, *CFLAGS, "-shared", SYNTH_SRC, "-o", SYNTH_LIB]
    all_jobs = jobs + ([synth_job] if synth_job else [])
    if all_jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
            for out in ex.map(_run, all_jobs):
                if verbose and out.strip():
                    print(out)
    if jobs or _stale(LIB, objs):
        _run([cc, *ARCH, "-shared", "-o", LIB, *objs])
    if os.path.exists(HOOKS_SRC) and (jobs or _stale(HOOKS_LIB, objs + [hooks_obj])):
        _run([cc, *ARCH, "-shared", "-o", HOOKS_LIB, *objs, hooks_obj])


if __name__ == "__main__":
    build(verbose=True, ptxas_verbose="-v" in sys.argv)
    print("built", LIB, SYNTH_LIB)
