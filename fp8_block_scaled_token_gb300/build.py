"""Build libfp8bs.so in-tree for sm_103a with nvcc (no cmake, no torch
extension machinery).  Each .cu file is one translation unit; they compile in
parallel and link into fp8_block_scaled_token_gb300/lib/libfp8bs.so with the
CUDA runtime linked statically.  The same sources built with -DFP8BS_DEBUG
(device-side bounds checks in the GEMM kernel) link into libfp8bs_debug.so.
Rebuilds only what is older than its sources."""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libfp8bs.so")
DEBUG_LIB = os.path.join(LIBDIR, "libfp8bs_debug.so")
# variant -> (extra nvcc flags, object directory, library)
VARIANTS = {
    "release": ([], OBJ, LIB),
    "debug": (["-DFP8BS_DEBUG"], os.path.join(OBJ, "debug"), DEBUG_LIB),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libfp8bs.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra, objdir):
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if r.stderr.strip():
            sys.stderr.write(r.stderr)
    return obj


def _link(objs, lib):
    if _stale(lib, objs):
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, variants=("release", "debug")) -> str:
    """Compile every .cu under csrc/ for each variant ("release" ->
    libfp8bs.so, "debug" -> libfp8bs_debug.so) in one parallel pool and link
    the libraries; return the release library's path."""
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = []
    for v in variants:
        flags, objdir, _ = VARIANTS[v]
        os.makedirs(objdir, exist_ok=True)
        if force:
            for o in glob.glob(os.path.join(objdir, "*.o")):
                os.remove(o)
        extra = flags + (["-Xptxas", "-v"] if verbose_ptxas else [])
        jobs += [(v, s, extra, objdir) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda j: (j[0], _compile(j[1], j[2], j[3])), jobs))
    for v in variants:
        _link([o for (vv, o) in objs if vv == v], VARIANTS[v][2])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                variants=("release",) if "--release-only" in sys.argv else ("release", "debug")))
