"""Build the CUDA library in-tree: paged_decode_attention_gb300/_build/libattn_decode.so.

One translation unit, one -gencode (sm_103a), no CMake; a few seconds with nvcc.
"""

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libattn_decode.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
GENCODE = "arch=compute_103a,code=sm_103a"


def _sources():
    out = []
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                out.append(os.path.join(d, f))
    return out


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return nvcc


def build(force=False, verbose=False):
    """Compile csrc/attn_decode.cu for sm_103a into _build/libattn_decode.so."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH):
        newest = max(os.path.getmtime(p) for p in _sources())
        if os.path.getmtime(LIB_PATH) >= newest:
            return LIB_PATH
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [
        _nvcc(), "-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17",
        "-Xcompiler", "-fPIC", "-shared", "-I", INCLUDE,
        "-o", tmp, os.path.join(CSRC, "attn_decode.cu"),
    ]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
