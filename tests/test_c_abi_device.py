"""The library driven from plain C99 on a GPU (tests/c_abi/device_check.c):
device buffers from cudaMalloc, a stream the program creates, and results
checked against values the ops' definitions fix, with no Python on the data
path."""
import os
import shutil
import subprocess

import pytest

from window_gather_swin_gb300 import build as lib_build

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_drives_the_library_on_the_gpu(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib = lib_build.build()
    exe = str(tmp_path / "device_check")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", "device_check.c"), "-o", exe, lib,
           "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "device ok", r.stdout + r.stderr
