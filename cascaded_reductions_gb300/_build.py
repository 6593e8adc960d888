"""Builds librf.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` file compiles to an object in parallel; the objects link
into ``cascaded_reductions_gb300/librf.so``.  A rebuild happens only when a
source or header is newer than the library.
"""

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librf.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills", "-I", INCLUDE, "-I", CSRC] + ARCH


def _nvcc():
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if p is None:
        raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")
    return p


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr


def build(force=False, verbose=False, extra_flags=(), lib=None, objdir=None):
    """Compile every CUDA source and link librf.so; returns the library path.

    ``lib`` / ``objdir`` build a variant elsewhere (e.g. the bounds-checked
    debug library, ``extra_flags=["-DRF_CHECK_BOUNDS"]``) without touching
    the default one."""
    lib = lib or LIB
    objdir = objdir or OBJDIR
    srcs = _sources()
    hdrs = _headers()
    if not force and not _stale(lib, srcs + hdrs):
        return lib
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)
    objs = [os.path.join(objdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    jobs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        for s, o in zip(srcs, objs):
            if force or _stale(o, [s] + hdrs):
                jobs.append(ex.submit(_compile, nvcc, s, o, list(extra_flags)))
        logs = [j.result() for j in jobs]
    if verbose:
        for lg in logs:
            if lg:
                print(lg)
    tmp = lib + ".tmp"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_checked(force=False):
    """The bounds-checked debug variant: _build_checked/librf_checked.so."""
    d = os.path.join(HERE, "_build_checked")
    return build(force=force, extra_flags=["-DRF_CHECK_BOUNDS"],
                 lib=os.path.join(d, "librf_checked.so"), objdir=d)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
