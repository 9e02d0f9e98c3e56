"""Builds libmoe_nvfp4.so (the product library) and libmoe_nvfp4_test.so (the test build)
in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel. The product library links the objects of
csrc/*.cu (CUDA runtime linked statically); the test library links the same objects plus
those of csrc/testbuild/*.cu, the entry points of include/moe_nvfp4_test.h, which only
tests load. The build is skipped when both libraries are newer than every source.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
TESTBUILD = os.path.join(CSRC, "testbuild")
LIB = os.path.join(PKG, "libmoe_nvfp4.so")
TEST_LIB = os.path.join(PKG, "libmoe_nvfp4_test.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--diag-suppress", "128", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_nvfp4.so")


def sources() -> list[str]:
    """The product library's translation units."""
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def test_sources() -> list[str]:
    """The test build's extra translation units."""
    return sorted(os.path.join(TESTBUILD, f) for f in os.listdir(TESTBUILD) if f.endswith(".cu"))


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if os.path.isfile(os.path.join(CSRC, f))]
    files += [os.path.join(TESTBUILD, f) for f in os.listdir(TESTBUILD)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return files


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(TEST_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(TEST_LIB))
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src: str) -> str:
        prefix = "test_" if os.path.dirname(src) == TESTBUILD else ""
        obj = os.path.join(BUILD, prefix + os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    product, extra = sources(), test_sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, product + extra))
    prod_objs, test_objs = objs[:len(product)], objs[len(product):]

    def link(out: str, objects: list[str]):
        tmp = out + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objects]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {out} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)

    link(LIB, prod_objs)
    link(TEST_LIB, prod_objs + test_objs)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
