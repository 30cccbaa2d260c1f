"""Build the CUDA library in-tree: bit_asymmetric_kv_kvq_gb300/_lib/libkvq.so.

One nvcc per translation unit, run in parallel, then one link.  Code is
generated for sm_103a only (GB300).  The C runtime is linked statically, so
the library needs only the CUDA driver at load time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIB = os.path.join(LIBDIR, "libkvq.so")
# the debug build: kernels check their buffer bounds, every cache buffer is followed by a canary
DEBUG_LIB = os.path.join(LIBDIR, "libkvq_debug.so")
DEBUG_OBJDIR = os.path.join(LIBDIR, "obj_debug")
DEBUG_FLAGS = ("-DKVQ_DEBUG_CHECKS",)

SOURCES = ["kvq_api.cpp", "kvq_quant.cu", "kvq_decode.cu", "kvq_decode_lut.cu", "kvq_decode_mma.cu", "kvq_noalloc.cu",
           "kvq_ablation.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libkvq.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "kvq.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib=None, objdir=None, csrc=None) -> str:
    """Build libkvq.so (or, with `lib`/`objdir`/`csrc`, a variant built elsewhere with extra nvcc flags)."""
    src_dir = csrc or CSRC
    target = lib or LIB
    odir = objdir or OBJDIR
    if not force and lib is None and not stale():
        return LIB
    nvcc = nvcc_path()
    os.makedirs(odir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", src_dir,
                     *extra_flags]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(odir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        cmd = [nvcc, *common, "-c", os.path.join(src_dir, src), "-o", obj]
        if src.endswith(".cu"):
            cmd.insert(1, "-Xptxas=-v") if verbose else None
        procs.append((src, cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, cmd, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out))
        elif verbose and out:
            sys.stderr.write(out)
    if failed:
        msg = "\n".join(f"--- {s} ---\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = target + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, target)
    return target


def build_debug(force: bool = False) -> str:
    """Build the debug variant (libkvq_debug.so) if it is missing or older than its sources."""
    if not force and os.path.exists(DEBUG_LIB) and all(os.path.getmtime(f) <= os.path.getmtime(DEBUG_LIB)
                                                        for f in _deps()):
        return DEBUG_LIB
    return build(force=True, extra_flags=DEBUG_FLAGS, lib=DEBUG_LIB, objdir=DEBUG_OBJDIR)


if __name__ == "__main__":
    if "--debug" in sys.argv:
        print(build_debug(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
