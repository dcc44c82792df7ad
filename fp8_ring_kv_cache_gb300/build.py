"""Build librc.so (the C ABI of include/rc.h) in-tree with nvcc for sm_103a,
and beside it librc_bounds.so, the same sources compiled with -DRC_BOUNDS_CHECK
(device-side index checks and guard zones around every buffer; see
rc_build_flags in rc.h).

Every .cu translation unit of both libraries compiles in parallel; each shared
library links the CUDA runtime statically.
Run: python fp8_ring_kv_cache_gb300/build.py [--force] [-v]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librc.so")
LIB_BOUNDS = os.path.join(HERE, "librc_bounds.so")
# (library, object directory, extra nvcc flags)
VARIANTS = [(LIB, OBJ, []), (LIB_BOUNDS, os.path.join(OBJ, "bounds"), ["-DRC_BOUNDS_CHECK"])]
SOURCES = ["rc_host.cu", "rc_write.cu", "rc_rotate.cu", "rc_attention.cu", "rc_noalloc.cu", "rc_window.cu",
           "rc_bf16.cu", "rc_fused.cu"]
HEADERS = ["rc_device.cuh", "rc_internal.h", "rc_layout.h"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _newest_dep() -> float:
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "rc.h"), __file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, objdir: str, extra: list[str]) -> str:
    obj = os.path.join(objdir, src.replace(".cu", ".o"))
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def _link(lib: str, objs: list[str]) -> None:
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Build what is out of date of librc.so and librc_bounds.so; returns librc.so's path."""
    newest = _newest_dep()
    todo = [v for v in VARIANTS if force or not os.path.exists(v[0]) or os.path.getmtime(v[0]) < newest]
    if not todo:
        return LIB
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    jobs = [(lib, objdir, src, flags + extra) for lib, objdir, flags in todo for src in SOURCES]
    for _, objdir, _ in todo:
        os.makedirs(objdir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[2], j[1], j[3]), jobs))
    for lib, _, _ in todo:
        _link(lib, [o for j, o in zip(jobs, objs) if j[0] == lib])
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
