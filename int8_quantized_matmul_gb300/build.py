"""Builds libi2s.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit under csrc/ is compiled by nvcc in parallel, then linked
into int8_quantized_matmul_gb300/_lib/libi2s.so with the CUDA runtime linked
statically and only the i2s_* / i8s_* symbols exported (so the library's own
runtime never interposes on another copy loaded in the same process).
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libi2s.so")
BUILD = os.path.join(HERE, "_build")

SOURCES = ["abi.cu", "quant.cu", "gemv_tc.cu", "gemm_tc.cu", "i8s.cu", "i8s_tc.cu", "i8s_elt.cu",
           "noalloc.cu"]
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-Xptxas", "-v"]


def _newest_input() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(os.path.dirname(HERE), "include", "i2s.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)

    def compile_one(src: str):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [NVCC, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, obj, r in results:
        log.append(f"== {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            sys.stderr.write("".join(log))
            raise RuntimeError(f"nvcc failed on {src}")
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("".join(log))
    if verbose:
        sys.stdout.write("".join(log))
    tmp = LIB + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for _, o, _ in results],
           "-Xlinker", f"--version-script={os.path.join(CSRC, 'exports.map')}", "-Xlinker", "-Bsymbolic"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
