"""Build step of libfused_logp.so (nvcc, sm_103a, in-tree).

Run ``python -m selected_token_logprob_gb300.build`` or call ``build()``.
The library is rebuilt when a source or the public header is newer than it.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libfused_logp.so")
SOURCES = [os.path.join(CSRC, "fused_logp.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("logp_kernels.cuh", "logp_prims.cuh",
                                                  "grpo_kernels.cuh", "linear_logp.cuh", "gemm_bf16.cuh")] + [os.path.join(INCLUDE, "fused_logp.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libfused_logp.so")


def command(out: str) -> list[str]:
    return [nvcc(), ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xptxas", "-v",
            "-I" + INCLUDE, "-Xcompiler", "-fPIC", "-shared", *SOURCES, "-o", out]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    tmp = f"{LIB}.tmp{os.getpid()}"
    res = subprocess.run(command(tmp), capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
