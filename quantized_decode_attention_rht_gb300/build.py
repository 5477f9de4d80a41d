"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Every translation unit under csrc/ is compiled in parallel, then linked into
``quantized_decode_attention_rht_gb300/libkvq.so``.  Objects live in ``_build/``
next to this file; a unit is recompiled only when it or a header is newer than
its object.  Run ``python -m quantized_decode_attention_rht_gb300.build``.

``build(variant="spintest")`` makes a TEST-ONLY library, ``libkvq_spintest.so`` (objects in
``_build_spintest/``), whose codebook decode kernel gives up a wait for its own bulk copies
after two non-blocking polls: the GPU test of the give-up path loads it to see the error
report on valid data.  The product never loads it."""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler",
              "-fvisibility=hidden", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "kvq.h")]


def _stale(src: str, obj: str, newest_header: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return os.path.getmtime(src) > t or newest_header > t


VARIANTS = {None: ([], "_build", "libkvq.so"), "spintest": (["-DKVQ_SPIN_TEST"], "_build_spintest", "libkvq_spintest.so")}


def _compile(nvcc: str, src: str, obj: str, verbose: bool, defines=()):
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return src, r.stderr


def build(verbose: bool = False, force: bool = False, variant=None) -> str:
    nvcc = _nvcc()
    defines, build_dir, lib_name = VARIANTS[variant]
    BUILD = os.path.join(HERE, build_dir)
    LIB = os.path.join(HERE, lib_name)
    os.makedirs(BUILD, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    newest_header = max(os.path.getmtime(h) for h in _headers())
    jobs = []
    objs = []
    for s in srcs:
        obj = os.path.join(BUILD, os.path.basename(s) + ".o")
        objs.append(obj)
        if force or _stale(s, obj, newest_header):
            jobs.append((s, obj))
    workers = max(1, min(len(jobs), os.cpu_count() or 4))
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            for src, log in ex.map(lambda j: _compile(nvcc, j[0], j[1], verbose, defines), jobs):
                if verbose and log:
                    sys.stderr.write(f"== {os.path.basename(src)}\n{log}")
    if force or jobs or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fvisibility=hidden"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
