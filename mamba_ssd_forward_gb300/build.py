"""Build libssd_gb300.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel to an object file in
_build/, then nvcc links them into mamba_ssd_forward_gb300/libssd_gb300.so.
Rebuilds only when a source or header is newer than the library.

build_debug() makes the debug-bounds variant libssd_gb300_debug.so (objects
in _build_debug/): the same sources compiled with SSD_DEBUG_BOUNDS defined,
so that every plain global access of the kernels checks its index against
its buffer's extent and reports a violation as SSD_ERR_BOUNDS.  It is a
testing aid, never the library the package loads.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libssd_gb300.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libssd_gb300_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssd_gb300")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          lib_path: str = LIB_PATH, build_dir: str = BUILD_DIR) -> str:
    """Compile every csrc/*.cu for sm_103a and link libssd_gb300.so."""
    if not force and not extra_flags and up_to_date(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=PKG)
    os.close(fd)
    try:
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return lib_path


def build_debug(force: bool = False, verbose: bool = False) -> str:
    """Compile the debug-bounds variant libssd_gb300_debug.so."""
    if not force and up_to_date(DEBUG_LIB_PATH):
        return DEBUG_LIB_PATH
    return build(force=True, verbose=verbose, extra_flags=["-DSSD_DEBUG_BOUNDS"],
                 lib_path=DEBUG_LIB_PATH, build_dir=DEBUG_BUILD_DIR)


if __name__ == "__main__":
    if "--debug-bounds" in sys.argv:
        print(build_debug(force="--force" in sys.argv, verbose="-v" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
