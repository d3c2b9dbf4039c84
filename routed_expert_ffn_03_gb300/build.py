"""Build the in-tree CUDA libraries for sm_103a (GB300).

``build()`` compiles every ``csrc/*.cu`` and ``csrc/*.cpp`` of the package into ``libmoe.so`` (the C ABI of
include/moe.h) and ``synth/csrc/synth_gen.cu`` into ``synth/libsynthgen.so`` (the
device fill of the seeded synthetic inputs).  Translation units compile in parallel;
a library is rebuilt only when a source or header is newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBMOE = os.path.join(PKG, "libmoe.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "csrc", "synth_gen.cu")
LIBSYNTH = os.path.join(ROOT, "synth", "libsynthgen.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return r


def build_moe(force: bool = False, verbose: bool = False) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    hdrs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "moe.h")]
    if not force and not _stale(LIBMOE, srcs + hdrs):
        return LIBMOE
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.splitext(os.path.basename(s))[0] + ".o")
        objs.append(o)
        jobs.append([nv] + ARCH + FLAGS + (["-Xptxas", "-v"] if verbose else []) + ["-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        for r in ex.map(_run, jobs):
            if verbose and r.stderr:
                print(r.stderr)
    tmp = LIBMOE + ".tmp.%d" % os.getpid()
    _run([nv] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread"])
    os.replace(tmp, LIBMOE)
    return LIBMOE


def build_synth(force: bool = False) -> str:
    if not force and not _stale(LIBSYNTH, [SYNTH_SRC]):
        return LIBSYNTH
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    tmp = LIBSYNTH + ".tmp.%d" % os.getpid()
    _run([nv] + ARCH + ["-O3", "-Xcompiler", "-fPIC", "-shared", SYNTH_SRC, "-o", tmp])
    os.replace(tmp, LIBSYNTH)
    return LIBSYNTH


def build(force: bool = False, verbose: bool = False):
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build_moe, force, verbose)
        b = ex.submit(build_synth, force)
        return a.result(), b.result()


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
