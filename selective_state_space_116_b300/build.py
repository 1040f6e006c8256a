"""Build the CUDA library in-tree: csrc/*.cu -> libssm_scan.so (sm_103a).

Run as ``python -m selective_state_space_116_b300.build`` or through
``__graft_entry__.build()``.  nvcc cross-compiles, so no GPU is needed.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libssm_scan.so")
SOURCES = ["ssm_scan.cu"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-shared",
    "--expt-relaxed-constexpr",
]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return [f for f in files if f.endswith((".cu", ".cuh", ".h"))]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile the library if any source is newer than it; return its path."""
    if not force and os.path.exists(LIBRARY):
        built = os.path.getmtime(LIBRARY)
        if all(os.path.getmtime(f) <= built for f in _deps()):
            return LIBRARY
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-o", tmp,
           *[os.path.join(CSRC, s) for s in SOURCES]]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
