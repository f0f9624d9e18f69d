"""Build libmsa.so in-tree: nvcc, sm_103a only, translation units in parallel.

    python -m block_sparse_gqa_msa_gb300.build
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmsa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """The product library, libmsa.so."""
    return _build(BUILD, LIB, [], force, verbose)


def build_starve(force: bool = False, verbose: bool = False) -> str:
    """A TEST-ONLY variant of the library, never used by the product: bounded
    pipeline waits give up after 2 ms instead of 1 s, and msa_test_starve(k)
    makes CTA 0 of one kernel leave out its first Q tile, so that the tests
    can drive the timeout path.  Built into _build/starve/."""
    d = os.path.join(BUILD, "starve")
    return _build(d, os.path.join(d, "libmsa_starve.so"),
                  ["-DMSA_TEST_STARVE", "-DMSA_WAIT_TIMEOUT_NS=2000000ull"], force, verbose)


def _build(out_dir: str, lib: str, defines: list[str], force: bool, verbose: bool) -> str:
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [
        os.path.join(HERE, "..", "include", "msa.h")]
    objs = []
    jobs = []
    for src in sources:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *headers, __file__]):
            jobs.append([nvcc, *ARCH, *NVCC_FLAGS, *defines, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        run([nvcc, *ARCH, "-shared", "-o", lib, *objs, "-lcudart_static", "-ldl", "-lrt",
             "-lpthread"])
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
