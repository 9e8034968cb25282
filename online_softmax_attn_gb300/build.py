"""Compile the CUDA library for sm_103a, in-tree.

Produces ``online_softmax_attn_gb300/libattn_gb300.so`` from the ``csrc/*.cu``
translation units, compiled in parallel with nvcc (one ``-gencode``) and linked
with the static CUDA runtime, so the library needs no libcuda at load time
(driver entry points are resolved at run time).

    python -m online_softmax_attn_gb300.build [--force] [--ptxas-verbose] [--debug]

``--debug`` builds ``libattn_gb300_debug.so`` instead, compiled with
``-DATTN_DEBUG``: the kernels check their store indices and shared-memory
offsets, record ATTN_DEVERR_DEBUG_INDEX in the device error word on a failed
check and skip that access (nothing traps).
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libattn_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libattn_gb300_debug.so")

SOURCES = ["api.cu", "merge.cu", "decode.cu", "prefill_simt.cu", "prefill_tc.cu",
           "decode_static.cu", "host_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    for cand in ("/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, ptxas_verbose: bool, debug: bool = False) -> str:
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
    if debug:
        cmd.append("-DATTN_DEBUG")
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stderr if ptxas_verbose else ""


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True,
          debug: bool = False) -> str:
    """Compile (if stale) and link the library (the -DATTN_DEBUG variant with
    ``debug``); returns its path."""
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    headers = _headers()
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(build_dir, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [src, *headers]):
            jobs.append((src, obj))
    logs = []
    if jobs:
        workers = min(len(jobs), max(1, os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            futs = [ex.submit(_compile, s, o, ptxas_verbose, debug) for s, o in jobs]
            for f in futs:
                logs.append(f.result())
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp"
        cmd = [nvcc_path(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib_path)
    if ptxas_verbose or not quiet:
        for log in logs:
            if log:
                sys.stderr.write(log)
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--debug", action="store_true", help="build the -DATTN_DEBUG variant")
    a = ap.parse_args(argv)
    print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False, debug=a.debug))


if __name__ == "__main__":
    main()
