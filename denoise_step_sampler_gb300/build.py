"""Build ``libdg.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  Usage: ``python -m denoise_step_sampler_gb300.build``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdg.so")

SOURCES = ["dg_api.cu", "dg_vocab.cu", "dg_canvas.cu", "dg_selfcond.cu", "dg_noalloc.cu",
           "dg_anneal.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _compile(src: str, verbose_ptxas: bool, defines=()) -> str:
    tag = "_waittest" if defines else ""
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + tag + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(WAIT_TEST_LIB):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(WAIT_TEST_LIB))
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "dg.h")]
    return any(os.path.getmtime(d) > t for d in deps)


# A test build of the library (same sources) whose self-conditioning GEMM has
# a 1 ms bound on its pipeline waits and withholds the E copies of its third
# k-block, so that the MMA issuer's wait for them runs out: the bounded-wait
# exit path, tested without any fault.  Only the GEMM's object differs.
WAIT_TEST_LIB = os.path.join(HERE, "libdg_waittest.so")
WAIT_TEST_DEFINES = ["-DDG_WAIT_NS=1000000ull", "-DDG_TEST_WITHHOLD_E_STAGE=2"]


def _link(objs, out):
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """libdg.so and the wait test build libdg_waittest.so, if stale."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    jobs = [(s, []) for s in SOURCES] + [("dg_selfcond.cu", WAIT_TEST_DEFINES)]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose_ptxas, j[1]), jobs))
    _link(objs[:len(SOURCES)], LIB)
    test_objs = [o for src, o in zip(SOURCES, objs) if src != "dg_selfcond.cu"] + [objs[-1]]
    _link(test_objs, WAIT_TEST_LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
