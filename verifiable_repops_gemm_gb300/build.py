"""Builds librepops.so (the CUDA library behind include/repops.h) in-tree.

Every translation unit is compiled for sm_103a only, in parallel, with the
flags that fix the arithmetic: no FMA contraction (-fmad=false), no flush to
zero, IEEE division and square root.  Output: verifiable_repops_gemm_gb300/_build/.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "librepops.so")
# The checked build: every hot-path kernel tests each global access against
# its buffer's span and skips one outside it (REPOPS_ERR_BOUNDS), in place of
# a memory sanitizer.  Same sources, -DREPOPS_DEBUG_BOUNDS, its own objects.
OUT_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(OUT_CHECKED, "librepops_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
ARITH = ["-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true"]
NVCC_FLAGS = (["-O3", "-lineinfo", "-std=c++17"] + ARCH + ARITH +
              ["-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
               "-Xcompiler", "-fno-fast-math", "-I", INCLUDE, "-I", CSRC])


def nvcc() -> str:
    p = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build librepops")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(INCLUDE, "*.h")))


def _flag_string(extra=()) -> str:
    return " ".join(ARCH + ARITH + [f for f in extra if f.startswith("-D")])


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra, out_dir: str = OUT) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    deps = [src, __file__] + _headers()
    if not _stale(obj, deps):
        return obj
    tmp = obj + ".tmp.%d" % os.getpid()
    cmd = ([nvcc()] + NVCC_FLAGS + extra +
           ['-DREPOPS_BUILD_FLAGS="%s"' % _flag_string(extra), "-c", src, "-o", tmp])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (os.path.basename(src), r.stdout, r.stderr))
    os.replace(tmp, obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 0, checked: bool = False) -> str:
    """Compiles (incrementally) and links librepops.so -- or, with checked,
    the access-checking librepops_debug.so -- and returns its path."""
    out_dir, lib = (OUT_CHECKED, LIB_CHECKED) if checked else (OUT, LIB)
    os.makedirs(out_dir, exist_ok=True)
    if force:
        for f in glob.glob(os.path.join(out_dir, "*.o")):
            os.remove(f)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if checked:
        extra = extra + ["-DREPOPS_DEBUG_BOUNDS"]
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, out_dir), srcs))
    if _stale(lib, objs) or force:
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv))
