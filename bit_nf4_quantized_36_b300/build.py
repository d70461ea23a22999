"""Build libqlora.so (in-tree) with nvcc for sm_103a."""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB_PATH = os.path.join(HERE, "libqlora.so")
# the same sources with device-side bounds checks (QLORA_DEVICE_CHECKS): for tests and debugging
CHECKED_LIB_PATH = os.path.join(HERE, "libqlora_checked.so")
SRC_MAIN = os.path.join(HERE, "csrc", "libqlora.cu")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # IEEE division/rounding is part of the format definition: no fast math anywhere
    "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
    "-cudart", "shared", "-shared",
    "-Xlinker", "-rpath=/usr/local/cuda/lib64",
]


def _sources():
    return (glob.glob(os.path.join(HERE, "csrc", "*.cu")) + glob.glob(os.path.join(HERE, "csrc", "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def needs_build(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile libqlora.so, or with `checks` libqlora_checked.so (device-side bounds checks)."""
    path = CHECKED_LIB_PATH if checks else LIB_PATH
    if not force and not needs_build(path):
        return path
    tmp = path + ".tmp%d" % os.getpid()
    cmd = [NVCC, *NVCC_FLAGS, *(["-DQLORA_DEVICE_CHECKS"] if checks else []), "-o", tmp, SRC_MAIN]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.check_call(cmd)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force=True, verbose=True))
