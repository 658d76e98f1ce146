"""Builds the CUDA library ``_build/libpa.so`` for sm_103a (in-tree, no cmake).

Each translation unit under ``csrc/`` is compiled by nvcc in parallel, then linked
into one shared library with the CUDA runtime linked statically.  The library is
rebuilt only when a source or header is newer than it.  ``build(instrumented=True)``
builds ``_build/libpa_ts.so``, the same sources with -DPA_TIMESTAMPS (stage
timestamps for launch-gap measurement, see include/pa_timestamps.h).

    python -m paged_kv_decode_metadata_gb300.build [--force] [--ts]
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libpa.so")
TS_LIB_PATH = os.path.join(BUILD_DIR, "libpa_ts.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden visibility: the library exports only the C ABI (PA_API in include/pa.h).  Two
# builds loaded in one process (production and instrumented) then share no symbol --
# function-local statics of templates would otherwise be unified across libraries.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              f"-I{INCLUDE}", f"-I{CSRC}"]
# Keep the statically linked CUDA runtime's symbols local to the library.
LINK_FLAGS = ["-Xlinker", "--exclude-libs,ALL"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + glob.glob(os.path.join(INCLUDE, "*.h"))


def is_stale(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(src: str, extra=(), obj_dir: str = BUILD_DIR) -> str:
    obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, instrumented: bool = False) -> str:
    """Compile and link the library if needed; returns its path."""
    lib_path = TS_LIB_PATH if instrumented else LIB_PATH
    if not force and not is_stale(lib_path):
        return lib_path
    obj_dir = os.path.join(BUILD_DIR, "ts") if instrumented else BUILD_DIR
    os.makedirs(obj_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DPA_TIMESTAMPS"] if instrumented else [])
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, obj_dir), srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", *LINK_FLAGS, *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                instrumented="--ts" in sys.argv))
