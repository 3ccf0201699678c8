"""Builds libgqa_attn.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into ``gqa_attention_decode_gb300/libgqa_attn.so`` with the CUDA runtime linked
statically, so loading the library needs no CUDA driver (the driver is only
touched on the first call that uses a GPU).  A stamp of the sources, the flags
and the nvcc version skips rebuilding when nothing changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libgqa_attn.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
# The bounds-checked build: every kernel checks the index of each global store
# against its extent and records violations in the status word.
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libgqa_attn_debug.so")
DEBUG_FLAGS = ["-DGQA_DEBUG_BOUNDS"]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE, "-I", CSRC,
]
LINK_FLAGS = ARCH_FLAGS + ["-shared", "-cudart", "static", "-Xcompiler", "-fPIC"]


def nvcc_path() -> str:
    cands = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cands:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgqa_attn.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp(nvcc: str, extra: list[str]) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                h.update(f.encode())
                with open(os.path.join(d, f), "rb") as fh:
                    h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + extra + LINK_FLAGS).encode())
    h.update(subprocess.run([nvcc, "--version"], capture_output=True, text=True).stdout.encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link the library if needed; returns its path.  debug_bounds:
    the bounds-checked build (libgqa_attn_debug.so, objects apart)."""
    nvcc = nvcc_path()
    extra = DEBUG_FLAGS if debug_bounds else []
    lib_path = DEBUG_LIB_PATH if debug_bounds else LIB_PATH
    build_dir = os.path.join(BUILD_DIR, "debug") if debug_bounds else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    stamp = _stamp(nvcc, extra)
    stamp_file = os.path.join(build_dir, "libgqa_attn.stamp")
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib_path

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    r = subprocess.run([nvcc, *LINK_FLAGS, *objs, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
