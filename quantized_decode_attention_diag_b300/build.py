"""Build libkvq.so (sm_103a) in-tree with nvcc.

    python -m quantized_decode_attention_diag_b300.build [--verbose]

Compiles the CUDA kernels and the C-ABI host layer into one shared library next
to this file.  The CUDA runtime is linked statically, so the library needs only
the NVIDIA driver at run time (and not even that to load on a machine without
a GPU: only the calls that reach the device do).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libkvq.so")
SOURCES = ["kvq_api.cpp", "kvq_append.cu", "kvq_decode.cu", "kvq_static.cu", "kvq_calib.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvq.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cmd = [
        nvcc(), "-O3", "-std=c++17", ARCH, "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
        "-Xcompiler", "-ffp-contract=off", "-cudart", "static",
        "-I", INCLUDE, "-I", CSRC, "-o", LIB + ".tmp",
    ]
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stdout.write(res.stdout)
        sys.stderr.write(res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed with exit code {res.returncode}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(verbose="--verbose" in sys.argv, force=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
