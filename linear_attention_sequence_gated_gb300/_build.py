"""Build libgdn.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object in
``_build/``, then linked (static CUDA runtime) into ``libgdn.so`` beside this
file.  Nothing is installed.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
SOURCES = ["gdn_api.cu", "gdn_recurrent.cu", "gdn_chunked.cu", "gdn_attn.cu"]
HEADERS = [os.path.join(CSRC, "gdn_internal.h"), os.path.join(CSRC, "gdn_ptx.cuh"),
           os.path.join(os.path.dirname(PKG), "include", "gdn.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")
    return exe


def _newest_input(src: str) -> float:
    times = [os.path.getmtime(src)] + [os.path.getmtime(h) for h in HEADERS if os.path.exists(h)]
    return max(times)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    objs, procs = [], []
    for name in SOURCES:
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name.replace(".cu", ".o"))
        log = os.path.join(BUILD, name.replace(".cu", ".log"))
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < _newest_input(src):
            cmd = [exe] + NVCC_FLAGS + ["-c", src, "-o", obj]
            procs.append((name, log, subprocess.Popen(cmd, stdout=open(log, "w"),
                                                      stderr=subprocess.STDOUT)))
    failed = []
    for name, log, p in procs:
        if p.wait() != 0:
            failed.append((name, open(log).read()))
        elif verbose:
            print(open(log).read())
    if failed:
        msg = "\n".join(f"--- {n} ---\n{t}" for n, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or procs or not os.path.exists(LIB) or \
            os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([exe] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
