"""Compile the CUDA library ``libfa_gb300.so`` in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
the objects are linked into one shared library next to this file. The CUDA
runtime is linked statically, so loading the library needs no CUDA driver
until the first call that touches the GPU.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xptxas", "-v", "--expt-relaxed-constexpr"] + ARCH


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return (sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the library if any source is newer than it; return its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        log = obj + ".log"
        cmd = [nvcc, *NVCC_FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
        fh = open(log, "w")
        procs.append((src, obj, log, fh, subprocess.Popen(cmd, stdout=fh, stderr=subprocess.STDOUT)))
    failed = []
    for src, obj, log, fh, p in procs:
        p.wait()
        fh.close()
        if p.returncode != 0:
            failed.append((src, log))
        elif verbose:
            sys.stdout.write(open(log).read())
    if failed:
        msgs = []
        for src, log in failed:
            msgs.append(f"--- {os.path.basename(src)} ---\n" + open(log).read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    tmp = LIB + f".tmp{os.getpid()}"
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in sources()]
    subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
