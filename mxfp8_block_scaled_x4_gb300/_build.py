"""Build the CUDA library in-tree: mxfp8_block_scaled_x4_gb300/_lib/libmxfp8_gb300.so,
and its debug build libmxfp8_gb300_debug.so (compiled with MXFP8_DEBUG: every
computed global store index is checked against its buffer; the tests run it
in a process of its own).

Plain nvcc, one -gencode (sm_103a), all translation units of both builds
compiled in parallel, then one shared link each against the CUDA runtime.
No cmake.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(ROOT, "_build", "mxfp8")
OBJ_DEBUG = os.path.join(ROOT, "_build", "mxfp8_debug")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libmxfp8_gb300.so")
LIB_DEBUG = os.path.join(LIBDIR, "libmxfp8_gb300_debug.so")
SOURCES = ["api.cu", "quant.cu", "gemm.cu", "noalloc.cu", "moe.cu", "tactics.cu"]
HEADERS = ["ptx.cuh", "quant_block.cuh", "internal.h", "debug_check.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def _nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose=False):
    os.makedirs(OBJ, exist_ok=True)
    os.makedirs(OBJ_DEBUG, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + \
        [os.path.join(ROOT, "include", h) for h in ("mxfp8.h", "mxfp8_moe.h", "mxfp8_testing.h")]
    jobs = []
    links = []
    for objdir, lib, extra in ((OBJ, LIB, []), (OBJ_DEBUG, LIB_DEBUG, ["-DMXFP8_DEBUG"])):
        objs = []
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(objdir, src.replace(".cu", ".o"))
            objs.append(o)
            if force or _stale(o, [s] + hdrs):
                jobs.append([nvcc] + ARCH + FLAGS + extra + ["-I", os.path.join(ROOT, "include"), "-c", s, "-o", o])
        links.append((lib, objs))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), max(2, os.cpu_count() or 2))) as ex:
            list(ex.map(run, jobs))
    for lib, objs in links:
        if force or _stale(lib, objs):
            tmp = lib + ".%d.tmp" % os.getpid()
            run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs)
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
