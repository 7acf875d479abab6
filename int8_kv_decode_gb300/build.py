"""Build libkattn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel; the shared library links the CUDA
runtime statically so it does not depend on which libcudart the process
loaded first.  Object files go to ``_build/`` next to this file.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-ffp-contract=off",
          "-I", INCLUDE, "-I", CSRC]

# Per-file extra flags.  The exact-mode scan and the host constant generator
# must not contract multiply-add pairs.
SOURCES = {
    "kattn_api.cu": [],
    "quantize.cu": [],
    "qk_debug.cu": [],
    "decode_fast.cu": [],
    "decode_fast_paged.cu": [],
    "decode_tc.cu": [],
    "decode_noalloc.cu": [],
    "decode_exact.cu": ["--fmad=false"],
    "expf_constants.cu": ["--fmad=false"],
    "hash_rows.cu": [],
}


def nvcc_path() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: set NVCC or put the CUDA toolkit on PATH")


def _headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}")
    if verbose and r.stdout.strip():
        print(r.stdout, flush=True)
    return r.stdout


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile and link libkattn.so; returns its path.  Rebuilds what is stale."""
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    headers = _headers()
    jobs = []
    objs = []
    for src, extra in SOURCES.items():
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, __file__] + headers):
            cmd = [nvcc, "-c", s, "-o", o] + ARCH + COMMON + extra
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)
    outputs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            outputs = list(ex.map(lambda c: _run(c, verbose), jobs))
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + ".tmp"
        _run([nvcc, "-shared", "-o", tmp] + ARCH + objs + ["-cudart", "static"], verbose)
        os.replace(tmp, LIB)
    if ptxas_verbose:
        for out in outputs:
            print(out)
    return LIB


# Test-only build: exact mode's hand-off waits give up after this many polls
# (0: at once), so that a test can check the give-up path -- NaN rows and the
# KATTN_DEVERR_TIMEOUT bit -- with no wait that could block.  Never loaded by
# the package; only tests/test_gpu_exact_timeout.py loads it.
TIMEOUT_VARIANT_LIB = os.path.join(BUILD, "libkattn_exact_spin0.so")


def build_exact_timeout_variant(verbose: bool = False) -> str:
    """libkattn.so with decode_exact.cu built with KATTN_EXACT_SPIN_LIMIT = 0
    (every other object shared with the library); returns its path."""
    build(verbose=verbose)
    nvcc = nvcc_path()
    src = os.path.join(CSRC, "decode_exact.cu")
    obj = os.path.join(BUILD, "decode_exact_spin0.o")
    deps = [src, __file__] + _headers()
    if _stale(obj, deps):
        _run([nvcc, "-c", src, "-o", obj] + ARCH + COMMON + SOURCES["decode_exact.cu"]
             + ["-DKATTN_EXACT_SPIN_LIMIT=0u"], verbose)
    objs = [os.path.join(BUILD, f.replace(".cu", ".o")) for f in SOURCES if f != "decode_exact.cu"]
    if _stale(TIMEOUT_VARIANT_LIB, objs + [obj]):
        tmp = TIMEOUT_VARIANT_LIB + ".tmp"
        _run([nvcc, "-shared", "-o", tmp] + ARCH + objs + [obj, "-cudart", "static"], verbose)
        os.replace(tmp, TIMEOUT_VARIANT_LIB)
    return TIMEOUT_VARIANT_LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv)
    print(LIB)
