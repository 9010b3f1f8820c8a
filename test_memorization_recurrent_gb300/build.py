"""Build libatlasmem.so (sm_103a) in-tree with nvcc: one object per .cu file,
compiled in parallel, then linked into a shared library under _build/.

``build_variant`` builds a separately named copy with extra preprocessor
definitions (used by tests that need a test-only switch compiled in); the
library the package loads is always the plain one."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libatlasmem.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
         "-I", CSRC, "--expt-relaxed-constexpr"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "atlas_mem.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, objdir: str, extra) -> str:
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def _build(lib: str, objdir: str, extra, force: bool) -> str:
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, objdir, list(extra)), _sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, extra=()) -> str:
    return _build(LIB, OUT, extra, force)


def build_variant(name: str, defines, force: bool = False) -> str:
    """Build lib<name>.so under _build/<name>/ with -D<define> for each entry."""
    objdir = os.path.join(OUT, name)
    lib = os.path.join(objdir, f"lib{name}.so")
    return _build(lib, objdir, [f"-D{d}" for d in defines], force)


if __name__ == "__main__":
    print(build(force=True))
