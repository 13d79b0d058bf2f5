"""In-tree build of the CUDA library (sm_103a) and of the C input generator.

Every translation unit is compiled in parallel and linked into
``expert_cache_serving_gb300/_lib/libmoecache.so`` (CUDA runtime linked
statically, so the library loads without a GPU driver) and
``synth/_lib/libsynth.so``.
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
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libmoecache.so")
SYNTH_SRC = os.path.join(ROOT, "synth", "synth.c")
SYNTH_LIB = os.path.join(ROOT, "synth", "_lib", "libsynth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r


LAYER_INST = "layer_inst.cu"  # compiled once per (format, token bound)
SYNTH_GPU_SRC = os.path.join(ROOT, "synth", "synth_gpu.cu")
SYNTH_GPU_LIB = os.path.join(ROOT, "synth", "_lib", "libsynth_gpu.so")


def build_synth(verbose=False) -> str:
    os.makedirs(os.path.dirname(SYNTH_LIB), exist_ok=True)
    _run(["gcc", "-O3", "-fPIC", "-shared", "-ffp-contract=off", "-pthread", SYNTH_SRC, "-o", SYNTH_LIB], verbose)
    _run([_nvcc()] + ARCH + ["-O3", "-fmad=false", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static",
                             SYNTH_GPU_SRC, "-o", SYNTH_GPU_LIB], verbose)
    return SYNTH_LIB


DEBUG_LIBDIR = os.path.join(PKG, "_lib_debug")
DEBUG_LIB = os.path.join(DEBUG_LIBDIR, "libmoecache.so")


def build_cuda(verbose=False, debug=False) -> str:
    """debug: the bounds-checked build (-DMOE_DEBUG_BOUNDS) in _lib_debug/."""
    objdir = os.path.join(DEBUG_LIBDIR, "obj") if debug else OBJDIR
    lib = DEBUG_LIB if debug else LIB
    extra = ["-DMOE_DEBUG_BOUNDS"] if debug else []
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if not srcs:
        raise RuntimeError("no CUDA sources")
    # (source, extra defines, object): the decode layer kernel's source is
    # compiled once per (format, token bound) so its 15 instantiations build
    # in parallel
    units = []
    for s in srcs:
        base = os.path.basename(s)
        if base == LAYER_INST:
            for fmt in (0, 1, 2):
                for maxt in (1, 2, 4, 8, 16):
                    units.append((s, extra + [f"-DMOE_LAYER_FMT={fmt}", f"-DMOE_LAYER_MAXT={maxt}"],
                                  os.path.join(objdir, f"{base}.{fmt}.{maxt}.o")))
        else:
            units.append((s, extra, os.path.join(objdir, base + ".o")))
    objs = [o for _, _, o in units]
    workers = max(1, min(len(units), os.cpu_count() or 8))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        jobs = [ex.submit(_run, [nvcc] + ARCH + NVCC_FLAGS + defs + ["-c", s, "-o", o], verbose) for s, defs, o in units]
        for j in jobs:
            j.result()
    _run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", lib] + objs + ["-lpthread", "-ldl", "-lrt"], verbose)
    return lib


def build_all(verbose=False) -> None:
    build_synth(verbose)
    build_cuda(verbose)
