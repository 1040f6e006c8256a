"""Build the CUDA library in-tree: csrc/*.cu -> libssm_scan.so (sm_103a).

Run as ``python -m selective_state_space_116_b300.build`` or through
``__graft_entry__.build()``.  nvcc cross-compiles, so no GPU is needed.  The
translation units compile in parallel and are linked into one shared library.

The library embeds a hash of its sources and compiler flags (returned by its
``ssm_build_id()``); ``build()`` recompiles whenever the library on disk
carries another hash (or none), so a library built from other sources is
never reused.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libssm_scan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "--expt-relaxed-constexpr"]
LINK_FLAGS = [*ARCH, "-shared"]


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return sorted(f for f in files if f.endswith((".cu", ".cuh", ".h")))


def source_hash(extra_flags=()) -> str:
    """Hash of every source file, the compiler flags and any extra flags."""
    h = hashlib.sha256()
    for f in _deps():
        with open(f, "rb") as fh:
            h.update(os.path.relpath(f, ROOT).encode() + b"\0" + fh.read() + b"\0")
    h.update(" ".join([*COMPILE_FLAGS, *LINK_FLAGS, *extra_flags]).encode())
    return h.hexdigest()[:24]


def built_id(path: str = LIBRARY):
    """The build id embedded in the library at `path`, or None (missing, or a
    library that predates the id).  Queried in a child process so that this
    process never maps a library it may be about to replace."""
    if not os.path.exists(path):
        return None
    code = ("import ctypes,sys; l=ctypes.CDLL(sys.argv[1]); f=getattr(l,'ssm_build_id',None);"
            "f is not None and setattr(f,'restype',ctypes.c_char_p);"
            "print(f().decode() if f is not None else '')")
    try:
        out = subprocess.run([sys.executable, "-c", code, path], capture_output=True, text=True,
                             timeout=120)
    except (OSError, subprocess.TimeoutExpired):
        return None
    return out.stdout.strip() or None if out.returncode == 0 else None


DEBUG_LIBRARY = os.path.join(HERE, "libssm_scan_debug.so")


def build(force: bool = False, verbose: bool = False, extra_flags=(), jobs: int = 0,
          debug: bool = False) -> str:
    """Compile the library unless the one on disk was built from these exact
    sources and flags; return its path.  debug: the -DSSM_DEBUG build (device
    bounds checks recorded in the workspace header, see ssm_scan_fwd_status)
    into libssm_scan_debug.so, for SSM_SCAN_LIBRARY."""
    library = DEBUG_LIBRARY if debug else LIBRARY
    if debug:
        extra_flags = (*extra_flags, "-DSSM_DEBUG")
    want = source_hash(extra_flags)
    if not force and built_id(library) == want:
        return library
    nvcc = os.environ.get("NVCC", "nvcc")
    tmpdir = tempfile.mkdtemp(prefix="ssm_build_")
    try:
        def compile_one(src):
            obj = os.path.join(tmpdir, src[:-3] + ".o")
            cmd = [nvcc, *COMPILE_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", "-o", obj,
                   os.path.join(CSRC, src)]
            if src == "ssm_scan.cu":
                cmd.insert(1, f'-DSSM_BUILD_ID="{want}"')
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
            if verbose and res.stderr:
                print(res.stderr, file=sys.stderr)
            return obj

        n = jobs or max(1, min(len(sources()), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
            objs = list(ex.map(compile_one, sources()))
        tmp = library + f".tmp{os.getpid()}"
        cmd = [nvcc, *LINK_FLAGS, "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, library)
    finally:
        shutil.rmtree(tmpdir, ignore_errors=True)
    return library


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
