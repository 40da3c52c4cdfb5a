"""Build the CUDA codec library in-tree: agent_shared_compressed_gb300/libkvcodec.so.

One nvcc process per translation unit (run in parallel), sm_103a only, then
one link step.  No CMake.  The result is git-ignored and rebuilt on each
machine (the GPU hosts are aarch64; this file builds natively wherever it
runs).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvcodec.so")

SOURCES = ["kvp_host.cu", "kvpool_encode.cu", "kvpool_decode.cu", "cachecard.cu", "kvpool_noalloc.cu", "kvpool_attend.cu",
           "kvp_probe.cu"]
HEADERS = ["kvp_internal.cuh", "kvp_vec.cuh", "kvp_async.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "kvpool.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src, extra):
    obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link the library if it is missing or older than its sources."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OBJ_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs = []
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for src, obj, rc, out in ex.map(lambda s: _compile(s, extra), SOURCES):
            if rc != 0:
                raise RuntimeError("nvcc failed on %s:\n%s" % (src, out))
            if verbose and out.strip():
                print(out, file=sys.stderr)
            objs.append(obj)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
