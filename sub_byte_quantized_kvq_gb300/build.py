"""Build the CUDA library (libkvq.so) in-tree for GB300 (sm_103a) with nvcc.

Each translation unit compiles in its own nvcc process (in parallel); the
objects link into one shared library exporting the C ABI of include/kvq.h.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]
# The quantizer's arithmetic runs exactly as written (no fused multiply-add):
# its binary32 error bounds and its fp64 recomputations assume one rounding
# per operation, as the definition has.
PER_TU = {"kvq_quantize.cu": ["--fmad=false"]}
TUS = ["kvq_api.cu", "kvq_quantize.cu", "kvq_decode.cu", "kvq_decode_int4.cu", "kvq_decode_e2m1.cu",
       "kvq_decode_cb2.cu", "kvq_decode_tiered.cu", "kvq_decode_cb2s.cu",
       "kvq_decode_a3.cu", "kvq_decode_cb2g.cu", "kvq_noalloc.cu"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "kvq.h"))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_mtime():
        return LIB
    nvcc = _nvcc()

    def compile_one(tu: str) -> str:
        obj = os.path.join(BUILD, tu.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *COMMON, *PER_TU.get(tu, []), "-c", os.path.join(CSRC, tu), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {tu}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(TUS)) as ex:
        objs = list(ex.map(compile_one, TUS))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
