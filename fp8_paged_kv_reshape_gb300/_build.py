"""Build libkvfp8.so in-tree for sm_103a (nvcc, one -gencode, units compiled in parallel)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIB_DIR, "libkvfp8.so")
# test-only variant for the bounded-wait timeout test (never loaded by the package)
WITHHOLD_LIB = os.path.join(LIB_DIR, "libkvfp8_withhold.so")
WITHHOLD_DEFINE = "-DKVFP8_TEST_WITHHOLD_FIRST_CHUNK=1"
HEADER = os.path.join(ROOT, "include", "kvfp8.h")

SOURCES = ["kvfp8_api.cu", "reshape_and_cache.cu", "paged_decode.cu", "paged_decode_mixed.cu",
           "prefill_attention.cu", "dequant.cu", "decode_noalloc.cu"]
DEPS = ["kvfp8_device.cuh", "kvfp8_internal.h", "paged_decode_kernel.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-Xptxas", "-warn-spills",
]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the kvfp8 CUDA library cannot be built")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    inputs = [os.path.join(CSRC, f) for f in SOURCES + DEPS] + [HEADER, __file__]
    return any(os.path.getmtime(p) > t for p in inputs)


def _compile(nvcc: str, src: str, obj: str, defines=(), verbose: bool = False) -> str:
    extra = os.environ.get("KVFP8_NVCC_EXTRA", "").split()
    cmd = [nvcc, *NVCC_FLAGS, *extra, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def _link(nvcc: str, objs, lib: str) -> str:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if it is missing or older than its sources."""
    if not force and not _stale(LIB):
        return LIB
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda src: _compile(nvcc, src, os.path.join(OBJ_DIR, src.replace(".cu", ".o")),
                                                verbose=verbose), SOURCES))
    return _link(nvcc, objs, LIB)


def build_withhold_variant(verbose: bool = False) -> str:
    """A test-only copy of the library whose single-query decode kernels withhold the copy
    of every CTA's first chunk and give up any wait after about 1e5 cycles, so that the
    bounded-wait timeout path can be driven on a GPU with no copy ever in flight.  Built
    from the same sources (paged_decode.cu recompiled with one define, the other units
    reused); the package never loads it."""
    build(verbose=verbose)
    if not _stale(WITHHOLD_LIB):
        return WITHHOLD_LIB
    nvcc = _nvcc()
    wdir = os.path.join(OBJ_DIR, "withhold")
    os.makedirs(wdir, exist_ok=True)
    objs = [os.path.join(OBJ_DIR, src.replace(".cu", ".o")) for src in SOURCES]
    objs[SOURCES.index("paged_decode.cu")] = _compile(
        nvcc, "paged_decode.cu", os.path.join(wdir, "paged_decode.o"), (WITHHOLD_DEFINE,), verbose)
    return _link(nvcc, objs, WITHHOLD_LIB)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
