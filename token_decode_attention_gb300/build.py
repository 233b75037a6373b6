"""Build ``libdattn.so`` in-tree for sm_103a with nvcc.

Translation units compile in parallel; the shared object links the CUDA runtime
statically so it loads next to any PyTorch build.  ptxas register / spill
reports are kept in ``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdattn.so")
SOURCES = ["decode_streamk.cu", "decode_cluster.cu", "decode_cluster_paged.cu", "combine.cu",
           "split_calls.cu", "decode_noalloc.cu", "selftest.cu", "softmax.cu", "rope_append.cu",
           "dattn_api.cpp"]
HEADERS = ["dattn_internal.h", "ptx.cuh", "streamk.h", "merge.cuh", "decode_kernel.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found (CUDA toolkit required to build libdattn)")
    return path


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, "dattn.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime()


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for (_, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp,
           *[obj for obj, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
