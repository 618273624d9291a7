"""Builds libdspark.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

``python -m draft_sampling_verification_gb300.build`` or ``build()``.  Each
``csrc/*.cu`` file is compiled by its own nvcc process (in parallel), then the
objects are linked into ``_build/libdspark.so``.  Strict IEEE fp32: no
--use_fast_math, no flush-to-zero; the deterministic q path additionally uses
explicit round-to-nearest intrinsics so no contraction can change it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libdspark.so")
# the bounds-checked build (DSPARK_CHECKED): every checked index site tests
# its bound and counts failures (dspark_checked_status); for tests only
OUT_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(OUT_CHECKED, "libdspark_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "--extended-lambda", "--expt-relaxed-constexpr", "-ftz=false",
                     "-prec-div=true", "-prec-sqrt=true"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdspark")
    return exe


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          checked: bool = False) -> str:
    out_dir, lib = (OUT_CHECKED, LIB_CHECKED) if checked else (OUT, LIB)
    extra = ["-DDSPARK_CHECKED"] if checked else []
    os.makedirs(out_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    newest_header = _newest(headers)
    exe = nvcc()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(out_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s),
                                                                         newest_header):
            cmd = [exe] + NVCC_FLAGS + extra + (["-Xptxas", "-v"] if ptxas_info else []) + \
                  ["-c", s, "-o", o]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, jobs):
                if verbose or ptxas_info or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError("nvcc failed: " + " ".join(cmd))
    if force or jobs or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        tmp = lib + ".%d.tmp" % os.getpid()
        cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checked="--checked" in sys.argv))
