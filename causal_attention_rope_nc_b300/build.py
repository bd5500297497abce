"""Build the in-tree CUDA library ``libncattn.so`` for sm_103a with nvcc.

All kernels and the C ABI live in one translation unit (``csrc/nc_api.cu``
includes the kernel headers), compiled with
``-gencode arch=compute_103a,code=sm_103a``.  The CUDA runtime is linked
statically, so the library loads on a machine without a GPU (the driver is
only needed when a kernel is launched).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libncattn.so")
# the bounds-checked debug build (-DNC_CHECK): every raw global store and the
# decode kernels' raw cache loads are checked against the tensors the call
# registered; a stray access is skipped and recorded in the status word
LIB_CHECK = os.path.join(HERE, "libncattn_check.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2", "-shared",
    "--expt-relaxed-constexpr",
]


def _sources():
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + [os.path.join(INCLUDE, "ncattn.h")])


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECK if checked else LIB
    if not force and not needs_build(lib):
        return lib
    cmd = [NVCC, *FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", lib, os.path.join(CSRC, "nc_api.cu")]
    if checked:
        cmd[1:1] = ["-DNC_CHECK"]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    subprocess.run(cmd, check=True)
    return lib


def build_all(force: bool = False) -> None:
    """The library and its bounds-checked debug build."""
    build(force=force)
    build(force=force, checked=True)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, checked="--checked" in sys.argv)
    print(LIB_CHECK if "--checked" in sys.argv else LIB)
