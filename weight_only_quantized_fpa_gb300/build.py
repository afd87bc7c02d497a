"""Build libwo.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel, then linked into
``_build/libwo.so``.  CUDA runtime is linked statically; the driver entry
points the tensor-core kernel needs are fetched at run time through the
runtime, so the library has no link-time dependency on libcuda.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libwo.so")
# the index-checked debug build (-DWO_DEBUG_BOUNDS=1): every computed global
# index is checked against its buffer's extent, failures recorded, not
# trapped (csrc/wo_bounds.cuh); loaded instead of LIB when the environment
# sets WO_DEBUG_BOUNDS=1
BUILD_DEBUG_BOUNDS = os.path.join(BUILD, "debug_bounds")
LIB_DEBUG_BOUNDS = os.path.join(BUILD_DEBUG_BOUNDS, "libwo_debug_bounds.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwo")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
           if f.endswith((".cu", ".cuh", ".h"))]
    out.append(os.path.join(INCLUDE, "wo.h"))
    return out


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_bounds: bool = False) -> str:
    out_dir = BUILD_DEBUG_BOUNDS if debug_bounds else BUILD
    lib_path = LIB_DEBUG_BOUNDS if debug_bounds else LIB
    os.makedirs(out_dir, exist_ok=True)
    deps = _deps()
    if not force and not _stale(lib_path, deps):
        return lib_path
    cc = nvcc()
    flags = ARCH + NVCC_FLAGS + ["-I", INCLUDE] + (extra_flags or [])
    if debug_bounds:
        flags = flags + ["-DWO_DEBUG_BOUNDS=1"]

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr, flush=True)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
