"""Build the CUDA library libqmv.so in-tree for sm_103a.

Each .cu file is compiled by its own nvcc process (in parallel), then linked
into ``bit_weight_only_packed_gb300/_lib/libqmv.so``.  No fast-math: the
kernels rely on IEEE fp32 rounding.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libqmv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def cflags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str, deps) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [
        os.path.join(ROOT, "include", "qmv.h"), __file__]
    if not force and not extra and not _stale(LIB, deps):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmpdir = os.path.join(OUT_DIR, f"obj{os.getpid()}")
    os.makedirs(tmpdir, exist_ok=True)
    cc = nvcc()
    flags = cflags(extra)
    if os.environ.get("QMV_PTXAS_V"):
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(tmpdir, os.path.basename(src) + ".o")
        r = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp_lib = LIB + f".tmp{os.getpid()}"
    link = [cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp_lib, *objs,
            "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp_lib, LIB)
    shutil.rmtree(tmpdir, ignore_errors=True)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
