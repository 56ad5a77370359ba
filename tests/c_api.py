"""Build the plain-C user of the C ABI (tests/c/step_c_api.c) against
include/medusa.h, the in-tree libmedusa_gb300.so and the CUDA runtime."""
import glob
import os
import shutil
import subprocess

import pytest

from medusa_speculative_decoding_02_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "step_c_api.c")


def cuda_dirs():
    home = os.environ.get("CUDA_HOME") or os.path.dirname(os.path.dirname(mbuild.nvcc()))
    inc = os.path.join(home, "include")
    libs = [d for d in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets",
                                                                                "*", "lib"))
            if glob.glob(os.path.join(d, "libcudart.so*"))]
    if not libs:
        pytest.skip("no CUDA runtime library found")
    return inc, libs[0]


def build_c_program(out_dir) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = mbuild.build()
    inc, libdir = cuda_dirs()
    pkg = os.path.dirname(lib)
    exe = os.path.join(str(out_dir), "step_c_api")
    subprocess.run([cc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", inc, SRC, "-o", exe,
                    "-L", pkg, "-lmedusa_gb300", "-L", libdir, "-lcudart", "-lm",
                    f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{libdir}"], check=True)
    return exe
