"""Builds libbfp8.so in-tree (block_scaled_fp8_02_gb300/_build/) with nvcc for sm_103a.

Translation units compile in parallel; the library links the CUDA runtime
statically and reaches the driver's tensor-map encoder through the runtime's
driver entry-point query, so it needs nothing but the driver at run time.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libbfp8.so")
SOURCES = ["bfp8_api.cu", "bfp8_quant.cu", "bfp8_gemm_swap.cu", "bfp8_gemm_wide.cu",
           "bfp8_gemm_ext.cu", "bfp8_gemm_pair.cu", "bfp8_gemv.cu",
           "bfp8_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libbfp8 needs the CUDA toolkit to build")


def _deps() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*")) + [os.path.join(ROOT, "include", "bfp8.h")])


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          trace: bool = False, out: str | None = None) -> str:
    """Compile (if needed) and return the path of libbfp8.so.

    trace=True builds a separate timeline-tracing variant (kernels record
    %globaltimer at role milestones; see bfp8_trace_read) into `out`."""
    lib = out or LIB
    deps = _deps()
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if trace:
        extra += ["-DBFP8_TRACE"]
    tag = "_trace" if trace else ""

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(BUILD, src.replace(".cu", tag + ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}\n{r.stdout}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=jobs or len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose_ptxas:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            for (_, log), src in zip(results, SOURCES):
                f.write(f"==== {src}\n{log}\n")
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}\n{r.stdout}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
