"""In-tree build of libmoe.so and libmoe_debug.so (CUDA, sm_103a) with nvcc.

Each translation unit compiles in parallel into ``_build/``, then nvcc links
the shared library next to this file. A stamp records the source hash, the
flags and the host machine, so a copy moved to another architecture
rebuilds.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmoe.so")
# the same library with the device-side bounds checks of csrc/dbg.cuh
LIB_DEBUG = os.path.join(PKG, "libmoe_debug.so")

SOURCES = ["moe_api.cu", "kernels_gemm.cu", "kernels_gemm_pair.cu", "kernels_mlp_fused.cu",
           "kernels_route.cu", "kernels_align.cu"]
HEADERS = ["ptx.cuh", "internal.h", "launch.cuh", "align_block.cuh", "topk_warp.cuh", "act.cuh",
           "dbg.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# hidden visibility: only the MOE_API entry points of include/moe.h are
# exported, so two builds in one process share no internal symbol
FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC]


def lib_path(debug: bool = False) -> str:
    return LIB_DEBUG if debug else LIB


def _flags(debug: bool) -> list[str]:
    return FLAGS + (["-DMOE_DEBUG"] if debug else [])


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _digest(debug: bool = False) -> str:
    h = hashlib.sha256()
    for f in SOURCES + HEADERS:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(INCLUDE, "moe.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(_flags(debug)).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def up_to_date(debug: bool = False) -> bool:
    lib = lib_path(debug)
    if not (os.path.exists(lib) and os.path.exists(lib + ".stamp")):
        return False
    with open(lib + ".stamp") as fh:
        return fh.read().strip() == _digest(debug)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile libmoe.so (libmoe_debug.so with debug=True) if missing or
    stale; returns its path."""
    lib = lib_path(debug)
    if not force and not extra_flags and up_to_date(debug):
        return lib
    out_dir = os.path.join(ROOT, "_build", "libmoe_debug" if debug else "libmoe")
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = _flags(debug) + list(extra_flags)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(lib + ".stamp", "w") as fh:
        fh.write(_digest(debug))
    return lib


def build_all(force: bool = False) -> tuple[str, str]:
    """Both libraries, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        rel = ex.submit(build, force)
        dbg = ex.submit(build, force, False, (), True)
        return rel.result(), dbg.result()


if __name__ == "__main__":
    print(build_all(force=True))
