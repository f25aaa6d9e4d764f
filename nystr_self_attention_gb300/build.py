"""Compile libnystrom.so in-tree with nvcc for sm_103a (GB300).

Objects go to ``_build/<machine>/`` beside the package sources so that x86
and Arm builds never mix; the shared library lands in the package folder.
Translation units compile in parallel.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libnystrom.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, obj: str, extra: list[str]) -> tuple[str, str]:
    cmd = [nvcc(), *ARCH_FLAGS, *CFLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, force: bool = False, extra: list[str] | None = None) -> str:
    """Compile every csrc/*.cu that changed and link libnystrom.so."""
    extra = list(extra or [])
    bdir = os.path.join(ROOT, "_build", platform.machine())
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    newest_header = max((os.path.getmtime(h) for h in headers), default=0.0)
    jobs = []
    objs = []
    for src in srcs:
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header):
            jobs.append((src, obj))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for obj, log in ex.map(lambda j: _compile(j[0], j[1], extra), jobs):
            if verbose and log.strip():
                print(log)
    # cuBLAS for the module's two projection GEMMs, found through an rpath to
    # the toolkit that compiled the library
    cuda_lib = os.path.realpath(os.path.join(os.path.dirname(nvcc()), "..", "lib64"))
    cmd = [nvcc(), *ARCH_FLAGS, "-shared", "-o", LIB + ".tmp", *objs, "-L", cuda_lib, "-lcublas",
           "-Xlinker", "-rpath=" + cuda_lib]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    if verbose:
        print("built", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose=True)
