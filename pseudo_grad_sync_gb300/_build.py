"""In-tree build of libdiloco_sync.so for sm_103a (nvcc, no cmake).

Each .cu file compiles to an object in parallel, then nvcc links the shared
library against the shared CUDA runtime (the same one PyTorch loads).
"""
from __future__ import annotations

import fcntl
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdiloco_sync.so")
SOURCES = ["dl_host.cu", "dl_stats.cu", "dl_quantize.cu", "dl_merge.cu", "dl_sync.cu", "dl_ring.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _cuda_lib_dir():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(cuda, "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "diloco_sync.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with open(os.path.join(BUILD, ".lock"), "w") as fh:
        fcntl.flock(fh, fcntl.LOCK_EX)
        if not force and not stale():
            return LIB
        nvcc = _nvcc()
        flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                        "-I", CSRC]
        if verbose or os.environ.get("DL_PTXAS_VERBOSE"):
            flags += ["-Xptxas", "-v"]
        procs, objs = [], []
        for src in SOURCES:
            obj = os.path.join(BUILD, src.replace(".cu", ".o"))
            objs.append(obj)
            cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
        failed = []
        for cmd, p in procs:
            out, _ = p.communicate()
            if out and (p.returncode != 0 or verbose or os.environ.get("DL_PTXAS_VERBOSE")):
                sys.stderr.write(out)
            if p.returncode != 0:
                failed.append(" ".join(cmd))
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
        tmp = LIB + f".tmp{os.getpid()}"
        link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
                "-Xlinker", "-rpath," + _cuda_lib_dir()]
        subprocess.run(link, check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
