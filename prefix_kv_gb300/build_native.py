"""Build ``libbca_gb300.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Usage: ``python -m prefix_kv_gb300.build_native [--force] [--debug] [-v]``.  The
translation units are compiled in parallel.  The library is rebuilt when the
content hash of its inputs (every source and header, this script, the compiler
flags and the nvcc version) differs from the one recorded beside it, or when it
is missing; copying a library to another machine therefore never passes a stale
or foreign build off as current.

``debug=True`` builds ``libbca_gb300_debug.so`` with ``-DBCA_BOUNDS_CHECK``: every
TMA coordinate, computed-address store and workspace or cache index in the
kernels is checked against its extent before use; a failed check skips the
access and reports ``BCA_ERR_BOUNDS`` in the status word.  The release library
contains none of these checks.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libbca_gb300.so")
LIB_DEBUG = os.path.join(LIB_DIR, "libbca_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I" + INCLUDE]
DEBUG_FLAGS = ["-DBCA_BOUNDS_CHECK"]
UNITS = ["attn_fwd.cu", "sched_prep.cu", "cache_append.cu", "bca_api.cu", "prefill_noalloc.cu", "selftest.cu",
         "qk_prologue.cu", "prefill_piecewise.cu", "page_pool.cpp"]
SOURCE_EXT = (".cu", ".cuh", ".h", ".cpp", ".hpp")


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(SOURCE_EXT)]
    out += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(SOURCE_EXT)]
    return sorted(out)


def _fingerprint(nvcc: str, debug: bool) -> str:
    """Content hash of everything the library is built from."""
    h = hashlib.sha256()
    for path in _sources() + [os.path.abspath(__file__)]:
        h.update(os.path.relpath(path, ROOT).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    flags = ARCH + FLAGS + (DEBUG_FLAGS if debug else []) + UNITS
    h.update("\0".join(flags).encode())
    ver = subprocess.run([nvcc, "--version"], capture_output=True, text=True, errors="replace")
    h.update(ver.stdout.encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def _stamp(lib: str) -> str:
    return lib + ".sha256"


def _current(lib: str, fp: str) -> bool:
    if not os.path.exists(lib) or not os.path.exists(_stamp(lib)):
        return False
    with open(_stamp(lib)) as f:
        return f.read().strip() == fp


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build (if needed) and return the path of the release or the debug library."""
    nvcc = _nvcc()
    lib = LIB_DEBUG if debug else LIB
    fp = _fingerprint(nvcc, debug)
    if not force and _current(lib, fp):
        return lib
    build_dir = BUILD + ("_debug" if debug else "")
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    extra = DEBUG_FLAGS if debug else []

    def compile_one(unit):
        obj = os.path.join(build_dir, os.path.splitext(unit)[0] + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, unit), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True, errors="replace")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {unit}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_one, UNITS))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True, errors="replace")
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    with open(_stamp(lib), "w") as f:
        f.write(fp + "\n")
    return lib


def build_all(force: bool = False) -> None:
    """Build the release and the bounds-checked library side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build, force, False, d) for d in (False, True)]:
            f.result()


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
