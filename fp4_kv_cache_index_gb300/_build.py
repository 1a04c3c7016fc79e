"""Builds the CSA2 CUDA library (libcsa2.so) in-tree with nvcc for sm_103a,
and on request its bounds-checked variant (libcsa2_debug.so, -DCSA2_DEBUG:
every checked index outside its buffer is recorded in the device error word
and the access skipped)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcsa2.so")
DEBUG_BUILD = os.path.join(ROOT, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libcsa2_debug.so")
SOURCES = ["csa2_api.cu", "k_append.cu", "k_index.cu", "k_index_fp4.cu", "k_topk.cu", "k_attn.cu",
           "k_hsi.cu", "k_swa.cu"]
HEADERS = ["csa2_device.cuh", "csa2_kernels.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, *extra]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    bdir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "csa2.h")]
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DCSA2_DEBUG"] if debug else [])
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if force or ptxas_info or _stale(o, [s] + headers):
            jobs.append([nvcc(), *_flags(extra), "-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        res = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, res):
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath", "-Xlinker", cuda_lib_dir()]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_synth(force: bool = False) -> str:
    """Device twin of the seeded input generator (csa2_synth/gen.cu)."""
    src = os.path.join(ROOT, "csa2_synth", "gen.cu")
    out = os.path.join(ROOT, "csa2_synth", "libcsa2synth.so")
    if force or _stale(out, [src]):
        tmp = out + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
               "-cudart", "shared", "-o", tmp, src,
               "-Xlinker", "-rpath", "-Xlinker", cuda_lib_dir()]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
    print(build_synth(force="--force" in sys.argv))
