"""Build libq4gemv.so in-tree with nvcc (sm_103a only).

Each translation unit under csrc/ compiles in parallel to an object in
_build/, then nvcc links the shared library next to this file.  A rebuild
happens only when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libq4gemv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "q4gemv.h"),
                                                                 os.path.abspath(__file__)]


# Library variants: the product, and a bounds-checking build for tests (every checked
# shared- and global-memory index counted and skipped when out of range).
VARIANTS = {
    "": (LIB_PATH, BUILD_DIR, ()),
    "check": (os.path.join(HERE, "libq4gemv_check.so"), os.path.join(BUILD_DIR, "check"), ("-DQ4_BOUNDS_CHECK",)),
}


def stale(variant: str = "") -> bool:
    lib = VARIANTS[variant][0]
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    lib_path, build_dir, vflags = VARIANTS[variant]
    if not force and not stale(variant):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    extra_flags = (*vflags, *extra_flags)

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "-v" in sys.argv else (),
                variant="check" if "--check" in sys.argv else ""))
