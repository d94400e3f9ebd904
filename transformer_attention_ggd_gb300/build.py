"""Builds libbam_attn.so (sm_103a) in-tree with nvcc.

Each .cu translation unit is compiled in parallel, then linked into one
shared library with a static CUDA runtime.  No cmake, no torch extension
machinery: the library exports a plain C ABI (include/bam_attn.h).

``build(debug=True)`` makes libbam_attn_debug.so from the same sources with
BAM_DEBUG defined: device-side bounds checks on every plain bulk copy and
tiled store, reported through the status word (BAM_ERR_BOUNDS).
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
LIB = os.path.join(BUILD, "libbam_attn.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(BUILD, "libbam_attn_debug.so")
SOURCES = ["api.cu", "table.cu", "fwd.cu", "bwd.cu", "decode.cu", "decode_noalloc.cu",
           "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         f"-I{os.path.join(ROOT, 'include')}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(ROOT, "include", "bam_attn.h")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    out_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    flags = FLAGS + (["-DBAM_DEBUG"] if debug else [])
    os.makedirs(out_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "bam_attn.h"))
    exe = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        if force or _stale(obj, [os.path.join(CSRC, src)] + headers):
            cmd = [exe, *ARCH, *flags, "-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
            if verbose:
                cmd.append("-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr)
            os.replace(obj + ".tmp", obj)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> tuple:
    """The release and the debug library, built side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        rel = ex.submit(build, force)
        dbg = ex.submit(build, force, False, True)
        return rel.result(), dbg.result()


if __name__ == "__main__":
    import sys
    if "--debug" in sys.argv:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug=True))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
