"""Build the CUDA library ``libtxl_gb300.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel to an object file under
``_build/``; the objects link into a shared library next to this file.  A
rebuild happens only when a source or header is newer than the library.
``build(debug=True)`` builds ``libtxl_gb300_debug.so`` (objects under
``_build_debug/``) with -DTXL_DEBUG: the kernels' device-side index checks.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtxl_gb300.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libtxl_gb300_debug.so")

SOURCES = ["txl_api.cu", "relattn_tc.cu", "relattn_combine.cu", "relattn_decode.cu",
           "relattn_decode_mma.cu", "relattn_f32.cu", "relpos.cu", "mem.cu", "relattn_noalloc.cu",
           "project.cu", "relattn_bwd.cu"]
HEADERS = [os.path.join(CSRC, "kernels.h"), os.path.join(CSRC, "decode.h"),
           os.path.join(CSRC, "decode_common.cuh"), os.path.join(CSRC, "ptx.cuh"),
           os.path.join(INCLUDE, "txl.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtxl_gb300.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile (if needed) and return the path of ``libtxl_gb300.so`` (with
    ``debug``: ``libtxl_gb300_debug.so``, built with -DTXL_DEBUG)."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and not _stale(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC] + (["-DTXL_DEBUG"] if debug else [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + [
        "-cudart", "shared", "-L", libdir, "-Xlinker", f"-rpath,{libdir}"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
