"""Build ``libfos_softmax.so`` in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each ``csrc/*.cu`` is compiled to an object in ``_build/`` in parallel, then linked into the
shared library next to this file.  Rebuilds only when a source or header is newer than the
library.  ``-Xptxas -v`` output (registers, spills, shared memory per kernel) is kept in
``_build/ptxas.log``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfos_softmax.so")
SOURCES = ["fos_api.cu", "fos_fwd.cu", "fos_bwd.cu", "fos_sink.cu", "fos_host.cu", "fos_qk.cu",
           "fos_pv.cu", "fos_kvgrad.cu"]
HEADERS = [os.path.join(CSRC, "fos_device.cuh"), os.path.join(CSRC, "fos_internal.h"),
           os.path.join(CSRC, "fos_tc.cuh"),
           os.path.join(ROOT, "include", "fos_softmax.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is needed to build libfos_softmax")


DEBUG_LIB = os.path.join(PKG, "libfos_softmax_debug.so")


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, debug: bool = False) -> str:
    """Compile and link the library if needed; returns its path.  ``debug`` builds the variant
    whose kernels check their indices (FOS_DEBUG) as ``libfos_softmax_debug.so`` instead."""
    lib = DEBUG_LIB if debug else LIB
    if not force and not _stale(lib):
        return lib
    bdir = BUILD + ("_debug" if debug else "")
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    extra = ["-DFOS_DEBUG"] if debug else []

    def compile_one(src):
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        return obj, res.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        for obj, log in results:
            f.write(f"== {os.path.basename(obj)}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True))
