"""Builds ``_build/libpagedkv.so`` in-tree: the CUDA kernels for sm_103a and the host
block manager, linked against the static CUDA runtime (no libcuda link-time
dependency; the driver is reached at run time)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_SOURCES = ["pa_decode.cu", "pa_cache.cu", "pa_decode_noalloc.cu", "pa_prefill.cu"]
CPP_SOURCES = ["block_manager.cpp"]
HEADERS = ["pa_device.cuh", "pa_internal.h", "pa_tc.cuh"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    deps += [os.path.join(INCLUDE, "pagedkv.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, defines=(), build_dir=None) -> str:
    """Compile and link the library; returns its path.

    ``defines`` (e.g. ``["PA_DECODE_STAGES=2"]``) and ``build_dir`` produce a
    variant build elsewhere; the default build is ``_build/libpagedkv.so``.
    """
    bdir = build_dir or BUILD
    lib = os.path.join(bdir, "libpagedkv.so")
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC] + [f"-D{d}" for d in defines]
    jobs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = [nvcc, *ARCH, *common, "-lineinfo", "-Xcompiler", "-fPIC", "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose_ptxas:
            cmd[1:1] = ["-Xptxas", "-v"]
        jobs.append((cmd, src))
        objs.append(obj)
    for src in CPP_SOURCES:
        obj = os.path.join(bdir, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-c",
               os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, src))
        objs.append(obj)
    procs = [(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), src)
             for cmd, src in jobs]
    failed = []
    for p, src in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if text.strip():
            sys.stderr.write(f"--- {src}\n{text}")
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"compilation failed: {', '.join(failed)}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
