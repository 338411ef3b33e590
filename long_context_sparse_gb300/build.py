"""Build the CUDA library in-tree: one nvcc per translation unit, in
parallel, then one shared-object link.  sm_103a only; static CUDA runtime so
the library has no run-time dependency beyond the driver.

    python -m long_context_sparse_gb300.build
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdsa_gb300.so")
LIB_CHECKS = os.path.join(PKG, "libdsa_gb300_checks.so")
SOURCES = ["select.cu", "indexer.cu", "indexer_topk.cu", "attn_fwd_tc.cu", "attn_bwd.cu",
           "attn_bwd_tc.cu", "dsa_api.cu",
           "dsa_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "-I",
                os.path.join(ROOT, "include")]


def _nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile the library.  checks=True builds the debug variant
    (libdsa_gb300_checks.so, -DDSA_CHECKS): the kernels bounds-check their
    shared-memory, TMEM and global offsets, latch DSA_ERR_DEVICE_CHECK and
    skip the access."""
    build_dir = BUILD + ("_checks" if checks else "")
    lib = LIB_CHECKS if checks else LIB
    flags = FLAGS + (["-DDSA_CHECKS"] if checks else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
               if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "dsa.h"))
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc] + flags + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("build failed:\n" + " ".join(cmd) + "\n" +
                               r.stdout + r.stderr)
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out)
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checks="--checks" in sys.argv))
