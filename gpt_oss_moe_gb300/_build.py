"""Build the CUDA library ``libgpt_oss_moe.so`` in-tree with nvcc (sm_103a).

Each ``csrc/*.cu`` compiles to an object in parallel, then nvcc links the
shared library (static cudart; the driver API is reached at run time through
cudaGetDriverEntryPointByVersion, so the library does not link libcuda).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgpt_oss_moe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags():
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "moe.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


# Build variants: name -> (library, object folder, extra nvcc flags).
# "debug_bounds" checks the index of every store of the layer's kernels and
# skips (and reports, MOE_DEV_BOUNDS) one that falls outside its buffer.
VARIANTS = {
    "": (LIB, BUILD, []),
    "debug_bounds": (os.path.join(PKG, "libgpt_oss_moe_debug_bounds.so"),
                     os.path.join(BUILD, "debug_bounds"), ["-DMOE_DEBUG_BOUNDS"]),
    # "trace" records per-CTA phase timestamps (moe_trace_read)
    "trace": (os.path.join(PKG, "libgpt_oss_moe_trace.so"),
              os.path.join(BUILD, "trace"), ["-DMOE_TRACE"]),
}


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Compile and link; returns the library path.  Rebuilds when a source,
    a header or this script is newer than the library."""
    lib, build_dir, vflags = VARIANTS[variant]
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = _flags() + vflags + list(extra_flags)

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
