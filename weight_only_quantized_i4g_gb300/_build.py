"""Build libqgemv.so (the CUDA kernels and the C ABI) in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into ``weight_only_quantized_i4g_gb300/libqgemv.so``.  No fast-math flags:
the kernels rely on IEEE binary32 rounding and on denormals being kept.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqgemv.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall", "--expt-relaxed-constexpr",
           "-Xptxas", "-warn-spills"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(PKG, "..", "include", "*.h"))
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or ptxas_info or not _newer(o, [s, *headers]):
            cmd = [NVCC, *ARCH, *NVFLAGS, "-c", s, "-o", o]
            if ptxas_info:
                cmd[1:1] = ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode != 0:
                print(" ".join(cmd))
                print(r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or jobs or not _newer(LIB, objs):
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
        os.replace(tmp, LIB)
    return LIB


def _build_variant(units, define: str, build_dir: str, lib: str, what: str, verbose: bool = False) -> str:
    """Compile `units` with -D`define` into build_dir and link them with the
    normal build's objects of the other units into `lib`."""
    build(verbose=verbose)
    os.makedirs(build_dir, exist_ok=True)
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(PKG, "..", "include", "*.h"))
    objs, jobs = [], []
    for s in sources():
        name = os.path.basename(s)
        if name not in units:
            objs.append(os.path.join(BUILD, name[:-3] + ".o"))
            continue
        o = os.path.join(build_dir, name[:-3] + ".o")
        objs.append(o)
        if not _newer(o, [s, *headers]):
            jobs.append([NVCC, *ARCH, *NVFLAGS, "-D" + define, "-c", s, "-o", o])
    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda c: (c, subprocess.run(c, capture_output=True, text=True)), jobs))
    failed = [c[-3] for c, r in results if r.returncode != 0]
    for c, r in results:
        if verbose or r.returncode != 0:
            print(" ".join(c))
            print(r.stdout + r.stderr)
    if failed:
        raise RuntimeError("nvcc (%s) failed for: %s" % (what, ", ".join(failed)))
    if jobs or not _newer(lib, objs):
        tmp = lib + ".tmp%d" % os.getpid()
        # -Bsymbolic: the variant's own references (the error word's address
        # above all) bind to its own definitions even when libqgemv.so is
        # loaded into the same process first
        r = subprocess.run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
                            "-Xlinker", "-rpath,/usr/local/cuda/lib64", "-Xlinker", "-Bsymbolic"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed (%s):\n%s" % (what, r.stdout + r.stderr))
        os.replace(tmp, lib)
    return lib


# Translation units of the decode GEMVs: the bounds-checking build compiles
# these with -DQG_BOUNDS_CHECK (every index a kernel forms is guarded; a guard
# that fails records QG_EBOUNDS and skips its access) and links them with the
# normal objects of the other units.
BC_UNITS = ("cs_common.cu", "gemv_i4g.cu", "gemv_fp8b128.cu", "gemv_fp8ue8m0.cu", "gemv_mq4v2.cu", "gemv_mq4v1.cu",
            "gemv_mq4c.cu", "gemv_q2_0.cu", "noalloc.cu")
BUILD_BC = os.path.join(PKG, "_build_bc")
LIB_BC = os.path.join(PKG, "libqgemv_bc.so")


def build_bounds_check(verbose: bool = False) -> str:
    """libqgemv_bc.so: the library with index guards in its decode GEMVs (for
    tests; slower than libqgemv.so, same results)."""
    return _build_variant(BC_UNITS, "QG_BOUNDS_CHECK", BUILD_BC, LIB_BC, "bounds-checking build", verbose)


# The stamps build (profiling): the error word's unit, the decode GEMVs of
# fmt=4, fmt=7 and MQ4-V2 and the no-allocation entry point compiled with
# -DQG_STAMPS, whose staged and warp-MMA kernels then record each block's
# timeline (qg_stamps_take).
STAMP_UNITS = ("cs_common.cu", "gemv_i4g.cu", "gemv_fp8b128.cu", "gemv_mq4v2.cu", "noalloc.cu")
BUILD_ST = os.path.join(PKG, "_build_st")
LIB_ST = os.path.join(PKG, "libqgemv_stamps.so")


def build_stamps(verbose: bool = False) -> str:
    """libqgemv_stamps.so: the library whose decode GEMVs stamp each block's
    timeline (for profiling; same results as libqgemv.so)."""
    return _build_variant(STAMP_UNITS, "QG_STAMPS", BUILD_ST, LIB_ST, "stamps build", verbose)


if __name__ == "__main__":
    import sys
    if "--bounds-check" in sys.argv:
        print(build_bounds_check(verbose="-v" in sys.argv))
    elif "--stamps" in sys.argv:
        print(build_stamps(verbose="-v" in sys.argv))
    else:
        print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_info="--ptxas" in sys.argv))
