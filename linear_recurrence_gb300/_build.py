"""Build libsscan.so (the sm_103a kernels and their C ABI) in-tree with nvcc.

Each translation unit compiles in parallel to ``_build/*.o`` and the objects
link into ``linear_recurrence_gb300/libsscan.so`` (CUDA runtime linked
statically, so the library needs only the driver at run time).  A build is
skipped when the library is newer than every source and header.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsscan.so")
UNITS = ["sscan_abi.cu", "sscan_fold.cu", "sscan_probe.cu", "sscan_noalloc.cu", "sscan_step.cu", "sscan_bwd.cu", "sscan_fwd_tma.cu"] + [
    f"sscan_fwd_tma_{dt}_{var}.cu" for dt in ("f32", "bf16") for var in "eoz"] + [
    f"sscan_fwd_shfl_{dt}.cu" for dt in ("f32", "bf16")] + [
    f"sscan_fwd_{dt}_{part}_{var}.cu" for dt in ("f32", "bf16") for part in "ab" for var in "eoz"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsscan.so")


def _inputs():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def compile_flags(verbose_ptxas: bool = False):
    flags = ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
             "-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    if not force and not verbose_ptxas and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = compile_flags(verbose_ptxas)

    def one(unit):
        src = os.path.join(CSRC, unit)
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        r = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=jobs or len(UNITS)) as ex:
        results = list(ex.map(one, UNITS))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", *ARCH, "-o", tmp, *[o for o, _ in results]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
