"""Build the CUDA library in-tree with nvcc for sm_103a only.

Output: dense_attention_forward_attn_gb300/_lib/libattn_fwd_<machine>.so, a
plain shared library exporting the C ABI of include/attn_fwd.h.  One
translation unit, one -gencode, no cmake.
"""
from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "_lib")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def lib_path(variant: str = "") -> str:
    suffix = f"_{variant}" if variant else ""
    return os.path.join(LIB_DIR, f"libattn_fwd{suffix}_{platform.machine()}.so")


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _sources():
    return ([os.path.join(CSRC, "attn_fwd.cu")] + glob.glob(os.path.join(CSRC, "*.cuh")) +
            [os.path.join(ROOT, "include", "attn_fwd.h")])


def build(force: bool = False, defines: dict | None = None, variant: str = "",
          verbose: bool = False) -> str:
    """Compile the library if any source is newer than it; return its path."""
    out = lib_path(variant)
    srcs = _sources()
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(s) for s in srcs)):
        return out
    os.makedirs(LIB_DIR, exist_ok=True)
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "lib64")
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-cudart", "shared", f"-Xlinker=-rpath,{cuda_lib}"]
    for k, v in (defines or {}).items():
        cmd.append(f"-D{k}={v}")
    if verbose:
        cmd += ["-Xptxas", "-v"]
    tmp = out + f".tmp{os.getpid()}"
    cmd += ["-o", tmp, os.path.join(CSRC, "attn_fwd.cu")]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
