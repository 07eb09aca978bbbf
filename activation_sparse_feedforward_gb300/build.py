"""Build ``libtwell.so`` (the C-ABI library) in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel, then linked
into ``activation_sparse_feedforward_gb300/libtwell.so``. The CUDA runtime is linked
statically and the driver is reached through ``cudaGetDriverEntryPointByVersion``,
so loading the library needs no GPU (symbol checks work on a CPU-only machine).

    python -m activation_sparse_feedforward_gb300.build [--verbose-ptxas] [--check]

``--check`` builds the bounds-checked variant ``libtwell_check.so`` (every kernel
compiled with -DTW_CHECK: indices computed from data are compared with their
buffers' sizes, and a violation raises TW_EBOUNDS instead of touching memory).
Select it at run time with TW_LIB_PATH=<path of libtwell_check.so>.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libtwell.so")
CHECK_BUILD_DIR = os.path.join(PKG_DIR, "_build_check")
CHECK_LIB_PATH = os.path.join(PKG_DIR, "libtwell_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtwell.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose_ptxas: bool = False, jobs: int | None = None, check: bool = False) -> str:
    nvcc = _nvcc()
    build_dir = CHECK_BUILD_DIR if check else BUILD_DIR
    lib_path = CHECK_LIB_PATH if check else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                    "-DNDEBUG"]
    if check:
        flags.append("-DTW_CHECK")
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose_ptxas="--verbose-ptxas" in sys.argv, check="--check" in sys.argv))
