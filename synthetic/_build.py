"""Builds and loads the generator's shared library (gcc, in-tree)."""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gen.c")
OUT = os.path.join(HERE, "libsynth.so")


def build(force: bool = False) -> str:
    lock = os.path.join(HERE, ".build.lock")
    with open(lock, "w") as fh:
        fcntl.flock(fh, fcntl.LOCK_EX)
        if force or not os.path.exists(OUT) or os.path.getmtime(OUT) < os.path.getmtime(SRC):
            tmp = OUT + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                   "-o", tmp, SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, OUT)
    return OUT


def load_library():
    return ctypes.CDLL(build())
