"""Build the CUDA library libmoe_b300.so in-tree for sm_103a (nvcc, no GPU needed)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoe_b300.so")
# The same library with the kernels' device-side index checks compiled in (-DMOE_CHECKS): an
# offset, row or slot index outside its range is reported as MOE_ERR_DEVICE_CHECK and skipped.
LIB_CHECKED = os.path.join(HERE, "libmoe_b300_checked.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-shared", "-Xcompiler", "-fPIC",
]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + [os.path.join(HERE, "..", "include", "moe.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(lib: str, extra: list[str], verbose: bool):
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, *FLAGS, *extra, *(["-Xptxas", "-v"] if verbose else []), *sources(),
           "-o", tmp]
    subprocess.check_call(cmd)
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> str:
    """Builds libmoe_b300.so and its bounds-checked twin; returns the default library's path."""
    if force or _stale(LIB):
        _compile(LIB, [], verbose)
    if force or _stale(LIB_CHECKED):
        _compile(LIB_CHECKED, ["-DMOE_CHECKS"], verbose)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
