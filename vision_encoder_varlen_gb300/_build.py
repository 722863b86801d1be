"""Build libvitattn.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each translation unit under csrc/ compiles in parallel to an object file under
_build/, then nvcc links the shared library into _lib/. Rebuilds only when a
source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libvitattn.so")
# the same library with the failure-path test hook compiled in (tests only; never loaded by the product)
TEST_LIB = os.path.join(LIBDIR, "libvitattn_testhooks.so")
TEST_HOOK_SOURCES = ("api.cu",)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libvitattn")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def compile_flags(ptxas_info: bool = False) -> list:
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    return flags + (["-Xptxas", "-v"] if ptxas_info else [])


def compile_all(out_dir: str, ptxas_info: bool = False) -> list:
    """Compile every translation unit into out_dir in parallel; [(object path, compiler stderr)]."""
    nvcc = _nvcc()
    os.makedirs(out_dir, exist_ok=True)
    flags = compile_flags(ptxas_info)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        r = subprocess.run([nvcc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        return list(ex.map(compile_one, _sources()))


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(LIBDIR, exist_ok=True)
    results = compile_all(BUILD, ptxas_info)
    for obj, err in results:
        if verbose and err.strip():
            print(err, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def build_test_hooks() -> str:
    """Build TEST_LIB: the release objects, with the translation units that hold the test hook
    (TEST_HOOK_SOURCES) compiled again with VIT_TEST_HOOKS defined."""
    build()
    if os.path.exists(TEST_LIB) and os.path.getmtime(TEST_LIB) >= os.path.getmtime(LIB):
        return TEST_LIB
    nvcc = _nvcc()
    objs = []
    for src in _sources():
        name = os.path.basename(src)
        if name in TEST_HOOK_SOURCES:
            obj = os.path.join(BUILD, name + ".testhooks.o")
            r = subprocess.run([nvcc, *compile_flags(), "-DVIT_TEST_HOOKS", "-c", src, "-o", obj],
                               capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {name} (test hooks):\n{r.stderr}")
        else:
            obj = os.path.join(BUILD, name + ".o")
        objs.append(obj)
    tmp = TEST_LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed (test hooks):\n{r.stderr}")
    os.replace(tmp, TEST_LIB)
    return TEST_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
