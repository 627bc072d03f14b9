"""Build librq.so (the CUDA kernels and the C ABI) for sm_103a, in-tree.

Each .cu file compiles in parallel to an object in nvfp4_quant_gb300/_build/,
then nvcc links nvfp4_quant_gb300/lib/librq.so (CUDA runtime linked
statically).  Rebuilds only when a source or header is newer than the library.
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "librq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "-I" + CSRC, "-I" + INCLUDE]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


# The row-kernel translation units hold one instantiation per quantisation
# mode (rq::QuantMode, 0 .. 6); each mode is compiled as its own object, in
# parallel, with -DRQ_MODE=<mode>.
ROW_MODES = range(7)


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _jobs():
    jobs = []
    for src in sources():
        if os.path.basename(src).startswith("rq_norm_quant_"):
            jobs += [(src, ["-DRQ_MODE=%d" % m], ".m%d" % m) for m in ROW_MODES]
        else:
            jobs.append((src, [], ""))
    return jobs


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link librq.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job):
        src, defs, tag = job
        obj = os.path.join(BUILD, os.path.basename(src) + tag + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *defs, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    jobs = _jobs()
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, jobs))
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -z defs: a mode left out of the objects fails here, not at load time
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "-z", "-Xlinker", "defs", "-o",
           tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
