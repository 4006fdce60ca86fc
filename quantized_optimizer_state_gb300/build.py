"""Build ``libfo.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

The library is compiled from ``csrc/*.cu`` with IEEE-exact FP32 flags
(no contraction, IEEE division and square root, no flush to zero) so that the
kernels reproduce the arithmetic contract of ``include/fo.h`` bit for bit.
Translation units compile in parallel; the result lands next to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libfo.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["fo_api.cu", "fo_step.cu", "fo_step_adamw.cu", "fo_step_adamw_dev.cu", "fo_step_sgd.cu",
           "fo_step_lion.cu", "fo_codecs.cu", "fo_verify.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -Xcompiler -ffp-contract=off: the host code derives the per-step scalars in
# double (1 - lr*wd and so on), which the contract defines as separately
# rounded operations; gcc would contract them into fused multiply-adds on
# aarch64.
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
              "-Xptxas", "-warn-spills"]

_lock = threading.Lock()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fo.h"))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    with _lock:
        if not force and not is_stale():
            return LIB
        os.makedirs(BUILD_DIR, exist_ok=True)
        cc = nvcc()

        def compile_one(src):
            obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
            cmd = [cc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c",
                   os.path.join(CSRC, src), "-o", obj]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
            return obj

        with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
            objs = list(ex.map(compile_one, SOURCES))
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
