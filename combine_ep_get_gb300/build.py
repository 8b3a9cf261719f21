"""Build libep_get.so (the CUDA library behind include/ep_get.h) in-tree.

Each .cu under csrc/ is compiled for sm_103a in parallel with nvcc, then the
objects are linked into combine_ep_get_gb300/libep_get.so (static cudart).
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libep_get.so")
HEADERS = [os.path.join(ROOT, "include", "ep_get.h")] + glob.glob(os.path.join(CSRC, "*.cuh"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-Xptxas", "-v"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in sources() + HEADERS + [__file__])


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc] + ARCH + NVCC_FLAGS + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(sources())) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for obj, log in results:
            sys.stderr.write(log)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for obj, log in results:
            f.write(log)
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, defines, recompile=("dispatch.cu",)) -> str:
    """A test-only copy of the library: the files in `recompile` (or every
    source, for recompile="all") compiled again with `defines` (e.g.
    ["-DEP_WAIT_TIMEOUT_NS=1000000ull"]) and linked with the product build's
    other objects into _build/<name>/libep_get_<name>.so.  Never the product
    library: only tests load it, by path.  Rebuilt when a source, a header or
    the defines changed."""
    build()
    out_dir = os.path.join(BUILD, name)
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libep_get_%s.so" % name)
    stamp = os.path.join(out_dir, "defines.txt")
    want = " ".join(defines) + " | " + (recompile if isinstance(recompile, str) else " ".join(recompile))
    if (os.path.exists(lib) and os.path.exists(stamp) and open(stamp).read() == want
            and os.path.getmtime(lib) >= os.path.getmtime(LIB)
            and all(os.path.getmtime(f) <= os.path.getmtime(lib) for f in sources() + HEADERS + [__file__])):
        return lib
    nvcc = _nvcc()

    def obj_of(src):
        base = os.path.basename(src)
        if recompile != "all" and base not in recompile:
            return os.path.join(BUILD, base + ".o")
        obj = os.path.join(out_dir, base + ".o")
        cmd = [nvcc] + ARCH + NVCC_FLAGS + list(defines) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj

    with ThreadPoolExecutor(max_workers=len(sources())) as ex:
        objs = list(ex.map(obj_of, sources()))
    tmp = lib + ".tmp.%d" % os.getpid()
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-Xlinker", "-Bsymbolic", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(want)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
