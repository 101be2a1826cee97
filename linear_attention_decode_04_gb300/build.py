"""Build the CUDA library in-tree: ``lib/libkda_decode.so`` for sm_103a (and
``lib/libkda_decode_timeline.so``, the same code with the decode kernel's
per-CTA timeline compiled in, for diagnostics).

Plain nvcc, no cmake: one translation unit per ``csrc/*.cu`` compiled in
parallel, then linked into one shared library against the shared CUDA runtime
(the same ``libcudart.so.13`` torch loads).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG_DIR, "csrc")
OUT_DIR = os.path.join(PKG_DIR, "lib")
OBJ_DIR = os.path.join(PKG_DIR, "_build")
LIB = os.path.join(OUT_DIR, "libkda_decode.so")
# the same library with the decode kernel's per-CTA timeline compiled in
# (diagnostics only; bench.py --case timeline)
TIMELINE_LIB = os.path.join(OUT_DIR, "libkda_decode_timeline.so")
TIMELINE_SRC = "kda_decode.cu"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise FileNotFoundError("nvcc not found")


def cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _link(nv: str, target: str, objs: list[str]) -> None:
    tmp = target + f".tmp{os.getpid()}"
    libdir = cuda_lib_dir(nv)
    cmd = [nv, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-Xlinker", f"-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every csrc/*.cu and link the library (and its timeline
    variant); returns the library's path."""
    nv = nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(INCLUDE, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")))
    objs = [os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o") for s in sources]
    jobs = [(s, o, ()) for s, o in zip(sources, objs)]
    tl_src = os.path.join(CSRC, TIMELINE_SRC)
    tl_obj = os.path.join(OBJ_DIR, "kda_decode_timeline.o")
    jobs.append((tl_src, tl_obj, ("-DKDA_DECODE_TIMELINE",)))

    def compile_one(job):
        src, obj, defs = job
        if not force and not _stale(obj, [src] + headers + [__file__]):
            return ""
        cmd = [nv, *ARCH, *NVCC_FLAGS, *defs, "-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return r.stderr if not defs else ""

    with cf.ThreadPoolExecutor(max(1, len(jobs))) as ex:
        logs = list(ex.map(compile_one, jobs))
    if verbose:
        for lg in logs:
            if lg:
                print(lg)
    if force or _stale(LIB, objs):
        _link(nv, LIB, objs)
    tl_objs = [tl_obj if o.endswith(os.sep + "kda_decode.o") else o for o in objs]
    if force or _stale(TIMELINE_LIB, tl_objs):
        _link(nv, TIMELINE_LIB, tl_objs)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
