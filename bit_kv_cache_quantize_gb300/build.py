"""Build ``libkvarn.so`` in-tree with nvcc for sm_103a (no cmake, no torch).

The translation units are compiled in parallel and linked into a shared
library exporting exactly the C ABI of ``include/kvarn.h``.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libkvarn.so")
SOURCES = ["kvarn_abi.cu", "quantize.cu", "decode.cu", "multiquery.cu"]
HEADERS = ["common.cuh", "tcgen05.cuh", "params.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"] + ARCH


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


OUT_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(OUT_CHECK, "libkvarn_check.so")


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """The checked (debug) build: the same sources compiled with KVARN_CHECK,
    so that every global store, partial read and bulk-copy source is tested
    against its buffer first (an out-of-range access is skipped and reported
    as KVARN_DEV_ERR_BOUNDS).  A separate library, libkvarn_check.so; the
    tests load it in place of libkvarn.so."""
    return build(force, verbose, out=OUT_CHECK, lib=LIB_CHECK, extra=["-DKVARN_CHECK"])


def build(force: bool = False, verbose: bool = False, out: str = OUT, lib: str = LIB, extra=()) -> str:
    os.makedirs(out, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "kvarn.h")]
    nvcc = _nvcc()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(out, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            jobs.append(([nvcc] + NVCC_FLAGS + list(extra) + ["-c", s, "-o", o + ".tmp"], o))

    def run(job):
        cmd, o = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {o}:\n{r.stdout}\n{r.stderr}")
        os.replace(o + ".tmp", o)
        with open(o + ".log", "w") as f:
            f.write(r.stderr)
        return r.stderr

    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for log in ex.map(run, jobs):
                if verbose:
                    sys.stderr.write(log)
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
    if "--checked" in sys.argv:
        print(build_checked(force="--force" in sys.argv, verbose=True))
