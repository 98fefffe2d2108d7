"""Build the CUDA library libtg_gemm.so in-tree for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a), then linked into one shared
library next to this file. No torch extension machinery: the library exports
a plain C ABI (include/tg_gemm.h).
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
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtg_gemm.so")
# the debug build (device-side bounds checks, TG_DEBUG=1): same sources, its own objects
OBJDIR_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libtg_gemm_debug.so")
SOURCES = ["tg_api.cu", "k_tiled.cu", "k_tiled2.cu", "k_splitk.cu", "k_w4.cu", "k_w4r.cu", "k_attn.cu", "k_softmax.cu", "k_fill.cu", "k_epilogue.cu", "k_pad.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tg_gemm.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    """Compile and link libtg_gemm.so (or, with debug=True, libtg_gemm_debug.so with the
    device-side bounds checks); returns its path. Skips work when up to date."""
    lib_path = LIB_DEBUG if debug else LIB
    objdir = OBJDIR_DEBUG if debug else OBJDIR
    if not force and not extra and up_to_date(lib_path):
        return lib_path
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = CFLAGS + ARCH + (["-DTG_DEBUG=1"] if debug else []) + (extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-lineinfo"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else None
    print(build(force=True, verbose=v or bool(extra), extra=extra, debug="--debug" in sys.argv))
