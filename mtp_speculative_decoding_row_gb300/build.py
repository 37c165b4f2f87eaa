"""Build the CUDA library ``libmtprs.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` file is compiled to an object in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3``, then linked
into a shared library against the shared CUDA runtime (the same
``libcudart.so.13`` PyTorch loads).  Rebuilds only when a source or header
is newer than the library.

``build(debug=True)`` builds the checking variant ``libmtprs_debug.so``
(``-DMTP_DEBUG``: the device primitives check their shared-memory, bulk-copy,
DSMEM and TMEM accesses and print a line starting with ``MTP_DEBUG`` for
any that fails) in its own object folder; the tests load it explicitly.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmtprs.so")
DEBUG_BUILD_DIR = os.path.join(ROOT, "_build", "debug")
DEBUG_LIB = os.path.join(PKG, "libmtprs_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmtprs.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale(debug: bool = False) -> bool:
    lib = DEBUG_LIB if debug else LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libmtprs.so (debug: libmtprs_debug.so) if needed;
    returns its path."""
    lib = DEBUG_LIB if debug else LIB
    bdir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and not is_stale(debug):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    flags = NVCC_FLAGS + (["-DMTP_DEBUG"] if debug else [])
    for src in _sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        log = obj + ".log"
        objs.append(obj)
        cmd = [cc, *flags, "-c", src, "-o", obj]
        procs.append((cmd, log, subprocess.Popen(cmd, stdout=open(log, "w"), stderr=subprocess.STDOUT)))
    failed = []
    for cmd, log, p in procs:
        if p.wait() != 0:
            failed.append((cmd, log))
        elif verbose:
            sys.stdout.write(open(log).read())
    if failed:
        msgs = "\n".join(" ".join(c) + "\n" + open(l).read() for c, l in failed)
        raise RuntimeError("nvcc failed:\n" + msgs)
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.check_call([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
