"""Builds libdflash2.so (and the test-hook library libdflash2_testing.so,
linked against it) in-tree with nvcc for sm_103a.

The translation units compile in parallel into ``_build/`` next to this file
and link into the two libraries beside it.  A unit is rebuilt when it or any
header is newer than its object.
"""

import concurrent.futures
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdflash2.so")

SOURCES = ["api.cu", "gemm_tc.cu", "gemm_simt.cu", "elementwise.cu", "attention.cu", "attention_tc.cu",
           "topk.cu", "selector.cu", "verify.cu", "select_static.cu"]
# the test hooks (include/dflash2_testing.h) live in a library of their own,
# linked against libdflash2.so, so the product library exports only dflash2.h
TEST_SOURCES = ["testing.cu"]
TEST_LIB = os.path.join(PKG, "libdflash2_testing.so")
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "internal.h"),
           os.path.join(ROOT, "include", "dflash2.h"), os.path.join(ROOT, "include", "dflash2_testing.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                "-I" + os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libdflash2.so")


def _stale(src, obj):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + HEADERS)


def _compile(src, verbose):
    obj = os.path.join(OBJ, os.path.splitext(os.path.basename(src))[0] + ".o")
    if not _stale(src, obj):
        return obj, False
    cmd = [nvcc()] + FLAGS + ["-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stdout + r.stderr)
    return obj, True


def _link(lib, objs, rebuilt, extra=()):
    if rebuilt or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + list(extra)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)


def build(verbose=False, jobs=None):
    """Compile and link libdflash2.so and the test-hook library beside it;
    returns the path of libdflash2.so."""
    os.makedirs(OBJ, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES + TEST_SOURCES]
    jobs = jobs or min(len(srcs), max(2, os.cpu_count() or 2))
    with concurrent.futures.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    n = len(SOURCES)
    objs = [o for o, _ in results[:n]]
    _link(LIB, objs, any(b for _, b in results[:n]))
    tobjs = [o for o, _ in results[n:]]
    _link(TEST_LIB, tobjs, any(b for _, b in results[n:]) or os.path.getmtime(LIB) > os.path.getmtime(TEST_LIB)
          if os.path.exists(TEST_LIB) else True,
          ["-L" + PKG, "-ldflash2", "-Xlinker", "-rpath=$ORIGIN"])
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
