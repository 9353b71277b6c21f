"""Build the CUDA library libfp8kv.so for sm_103a, in-tree.

Each .cu file is compiled to an object in parallel, then linked into
fp8_quantized_kv_gb300/_build/libfp8kv.so.  Objects are rebuilt only when a
source or header is newer.
"""
import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libfp8kv.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, extra, out_dir):
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        tmp = obj + f".tmp{os.getpid()}"
        cmd = [NVCC] + ARCH + FLAGS + extra + ["-c", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, trace: bool = False) -> str:
    """Build libfp8kv.so (or, with trace=True, libfp8kv_trace.so: the same
    library with per-tile clock stamps of one CTA of the tensor-core decode
    kernel, read with fp8kv_trace_read)."""
    out_dir = OUT + "_trace" if trace else OUT
    lib = os.path.join(out_dir, "libfp8kv_trace.so" if trace else "libfp8kv.so")
    os.makedirs(out_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if force:
        for o in glob.glob(os.path.join(out_dir, "*.o")):
            os.remove(o)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if trace:
        extra = extra + ["-DFP8KV_TRACE"]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, out_dir), srcs))
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, trace="--trace" in sys.argv))
