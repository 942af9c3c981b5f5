"""Builds the C-ABI shared library ``librlca.so`` in-tree with nvcc.

Each CUDA translation unit under ``csrc/`` is compiled for sm_103a in
parallel, then linked against the shared CUDA runtime (so the library and
PyTorch see the same current device and streams).  The same sources are
also built with ``-DRLCA_INDEX_CHECK`` into ``librlca_checked.so``, the
debugging build whose kernels check their indices (the tests run it).
Objects go to ``_build/`` at the repository root; the libraries land next
to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "librlca.so")
CHECKED_LIB = os.path.join(PKG, "librlca_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}", f"-I{CSRC}"] + ARCH


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build librlca.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _fingerprint(extra=()) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            h.update(f.encode())
            with open(os.path.join(d, f), "rb") as fh:
                h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


# the product library and the index-check build of the same sources
# (RLCA_INDEX_CHECK: every checked index that falls outside its array is
# recorded in a device status word and its access skipped; each call then
# waits for its kernels and returns RLCA_ERR_CUDA if one recorded anything)
VARIANTS = {
    "product": (LIB, os.path.join(BUILD, "obj"), []),
    "checked": (CHECKED_LIB, os.path.join(BUILD, "obj_checked"), ["-DRLCA_INDEX_CHECK"]),
}


def _stale(lib: str, stamp: str, fp: str) -> bool:
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return True
    with open(stamp) as f:
        return f.read().strip() != fp


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, variants=("product", "checked")) -> str:
    """Compile the libraries whose sources changed (all translation units of
    every variant in one parallel pool) and return the path of librlca.so."""
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    os.makedirs(BUILD, exist_ok=True)
    todo = []
    for name in variants:
        lib, objdir, flags = VARIANTS[name]
        stamp = os.path.join(BUILD, os.path.basename(lib) + ".stamp")  # build-cache fingerprint, not product source
        fp = _fingerprint(flags)
        if force or ptxas_info or _stale(lib, stamp, fp):
            os.makedirs(objdir, exist_ok=True)
            todo.append((lib, objdir, flags, stamp, fp))
    if not todo:
        return LIB
    srcs = _sources()

    def compile_one(job):
        src, objdir, flags = job
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + flags + extra + ["-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    # the slowest translation units first, so the pool's tail is short
    jobs = [(src, objdir, flags) for (lib, objdir, flags, _, _) in todo for src in srcs]
    jobs.sort(key=lambda j: -os.path.getsize(j[0]) if "k_" in os.path.basename(j[0]) else 0)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(compile_one, jobs))
    libdir = _cuda_lib_dir(nvcc)
    for lib, objdir, flags, stamp, fp in todo:
        objs = [os.path.join(objdir, os.path.basename(src)[:-3] + ".o") for src in srcs]
        tmp = lib + ".tmp"
        cmd = [nvcc, "-shared", "-cudart", "shared"] + ARCH + objs + [
            "-o", tmp, f"-L{libdir}", "-Xlinker", f"-rpath,{libdir}"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib)
        with open(stamp, "w") as f:
            f.write(fp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
