"""Build libg4.so in-tree for sm_103a with nvcc (no cmake, no torch extension machinery).

    python -m accelerator_decode_gb300.build
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libg4.so")
SOURCES = [os.path.join(HERE, "csrc", "g4.cu")]
DEPS = SOURCES + [os.path.join(HERE, "csrc", f) for f in ("common.cuh", "gemv.cuh", "gemv_s.cuh", "attn.cuh", "attn_mqa.cuh", "misc.cuh", "gemm_tc.cuh", "mega.cuh")]
DEPS.append(os.path.join(os.path.dirname(HERE), "include", "g4.h"))

NVCC_FLAGS = ["-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-shared", "-Xcompiler", "-fPIC"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def up_to_date():
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in DEPS if os.path.exists(p))


def build(force=False, verbose=False):
    if not force and up_to_date():
        return LIB
    tmp = LIB + ".tmp"
    cmd = [_nvcc()] + NVCC_FLAGS + ["-o", tmp] + SOURCES
    if verbose:
        print(" ".join(cmd), flush=True)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)
