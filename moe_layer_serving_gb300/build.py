"""Build libmegamoe.so (the C-ABI fused MoE library) for sm_103a, in tree.

Each .cu file compiles to an object in parallel, then one link; no cmake.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmegamoe.so")
# the same sources with the device-side bounds checks compiled in (MM_DEBUG):
# every indexed access of the SIMT stages and the GEMM tile decode is checked,
# a failed check latches MM_ERR_DEVICE with its site and skips the access
DEBUG_LIB = os.path.join(HERE, "libmegamoe_debug.so")
SOURCES = ["mm_api.cu", "mm_route.cu", "mm_gemm.cu", "mm_gemm2.cu", "mm_gemm16.cu", "mm_small.cu", "mm_noalloc.cu",
           "mm_ep.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "megamoe.h"))
    deps.append(__file__)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Build the release library and the bounds-checked debug library (both
    from the same sources, compiled in parallel); returns the release path."""
    targets = [(lib, flags) for lib, flags in ((LIB, []), (DEBUG_LIB, ["-DMM_DEBUG=1"]))
               if force or _stale(lib)]
    if not targets:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(job):
        src, tag, flags = job
        obj = os.path.join(BUILD, src.replace(".cu", f"{tag}.o"))
        cmd = [cc, *ARCH, *FLAGS, *flags, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    jobs = [(src, "" if lib == LIB else "_debug", flags) for lib, flags in targets for src in SOURCES]
    with cf.ThreadPoolExecutor(len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for i, (lib, _) in enumerate(targets):
        tmp = lib + f".{os.getpid()}.tmp"
        mine = objs[i * len(SOURCES):(i + 1) * len(SOURCES)]
        cmd = [cc, *ARCH, "-shared", "-o", tmp, *mine, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if v else []
    print(build(force=True, verbose=v, extra=extra))
