"""Builds the CUDA library ``_build/libpkv.so`` in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library with a C ABI (include/pkv.h).  ptxas register/spill reports go to
``_build/ptxas.log``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpkv.so")
UNITS = ["pkv_api.cu", "pkv_cache.cu", "pkv_merge.cu", "pkv_decode_simt.cu",
         "pkv_decode_simt_fp8.cu", "pkv_decode_mma.cu",
         "pkv_noalloc.cu", "pkv_prefill.cu", "pkv_prefill_tc.cu", "pkv_block_manager.cpp"]
HEADERS = ["pkv_common.cuh", "pkv_convert.cuh", "pkv_decode.cuh", "pkv_merge.cuh",
           "pkv_streamk.cuh", "pkv_prefill.cuh", "pkv_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the paged KV-cache library needs the CUDA toolkit")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(SRC, f) for f in UNITS + HEADERS]
    deps.append(os.path.join(os.path.dirname(PKG), "include", "pkv.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), out: str = None) -> str:
    """Compile (if stale) and return the path of libpkv.so.

    ``defines`` (e.g. ``["PKV_RING_BYTES_PER_WARP=16384"]``) and ``out`` build
    a variant library elsewhere (always rebuilt).
    """
    target = out or LIB
    if out is None and not defines and not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    tag = f"{os.getpid()}"

    def compile_unit(unit: str):
        obj = os.path.join(BUILD, os.path.splitext(unit)[0] + f".{tag}.o")
        cmd = [nvcc, *ARCH, *FLAGS, *[f"-D{d}" for d in defines], "-c",
               os.path.join(SRC, unit), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return unit, obj, r

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    log = []
    for unit, obj, r in results:
        log.append(f"==== {unit}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{r.stderr[-4000:]}")
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    os.makedirs(os.path.dirname(os.path.abspath(target)), exist_ok=True)
    tmp = target + f".{tag}.tmp"
    objs = [obj for _, obj, _ in results]
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"],
                       capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, target)
    if verbose:
        print(f"built {target}", file=sys.stderr)
    return target


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
