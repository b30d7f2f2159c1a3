"""include/wgs.h used from plain C99: the header compiles as C with
warnings as errors, a C program links against libwgs.so and its host-side
checks pass (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

from window_gather_swin_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_header_compiles_as_c_and_host_calls_behave(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib = lib_build.build()
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    exe = str(tmp_path / "abi_check")
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", cuda_inc,
           os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", exe,
           lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "abi ok", r.stdout + r.stderr
