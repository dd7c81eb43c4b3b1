"""The C ABI as a C or C++ user sees it, on the host (no GPU).

`include/diloco_sync.h` must compile as strict C99 and as C++17, and a plain
C program (`tests/c_abi_check.c`) must link against libdiloco_sync.so and run:
the version, status strings, the fragment planner on a worked LPT case,
workspace queries, and the refusals that validation returns before any
device work. The program is built in a scratch folder beside this file
(``tests/_cabi/``, ignored by git), which the test removes when it ends.
"""
from __future__ import annotations

import os
import shutil
import subprocess

from pseudo_grad_sync_gb300 import _build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
HEADER = os.path.join(INCLUDE, "diloco_sync.h")


def _cuda_lib_dir():
    nvcc = _build._nvcc()
    base = os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if os.sep in nvcc else \
        os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        d = os.path.join(base, sub)
        if os.path.isdir(d):
            return d
    return None


def test_header_compiles_as_c99_and_cpp17():
    for cmd in (["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                 "-x", "c", HEADER],
                ["g++", "-std=c++17", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                 "-x", "c++", HEADER]):
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_a_c_program_links_and_runs_the_host_side_abi():
    lib = _build.build()
    libdir = os.path.dirname(lib)
    work = os.path.join(HERE, "_cabi", str(os.getpid()))
    os.makedirs(work, exist_ok=True)
    try:
        exe = os.path.join(work, "c_abi_check")
        cmd = ["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
               os.path.join(HERE, "c_abi_check.c"), "-o", exe, "-L", libdir,
               f"-l:{os.path.basename(lib)}", f"-Wl,-rpath,{libdir}"]
        cuda = _cuda_lib_dir()
        if cuda:
            cmd += [f"-Wl,-rpath-link,{cuda}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        env = dict(os.environ)
        if cuda:
            env["LD_LIBRARY_PATH"] = os.pathsep.join(
                p for p in (cuda, env.get("LD_LIBRARY_PATH")) if p)
        r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
        assert r.returncode == 0 and r.stdout.strip() == "ok", (r.stdout, r.stderr)
    finally:
        shutil.rmtree(work, ignore_errors=True)
        try:
            os.rmdir(os.path.dirname(work))
        except OSError:
            pass
