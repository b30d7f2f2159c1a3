"""The residual rounding point, checked over all 2^32 binary16 pairs.

Page "BW1000 gfx936 Pangu-Weather inference profiling", s4, fixes
residual_out = fp16(fp32(residual) + fp32(branch)); the oracle rounds the
exact (double) sum once.  tests/pins/residual_pairs.c compares the oracle's
RN16(a + b) with the compiler's own binary32 add and binary16 conversion for
every ordered pair of bit patterns.  A stand-in library whose rounding is
toward zero must fail the same program, so the check has teeth.
"""
import os
import shutil
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "pins", "residual_pairs.c")

# A planted mistake: the oracle's decode, but rounding toward zero.
TRUNCATING = r"""
#include <stdint.h>
#include <string.h>
double orc_f16_to_f64(uint16_t u) { _Float16 h; memcpy(&h, &u, 2); return (double)h; }
uint16_t orc_rn16(double v) {
    _Float16 h = (_Float16)v;
    if (((double)h > v && v > 0) || ((double)h < v && v < 0)) {
        uint16_t u; memcpy(&u, &h, 2); u -= 1; return u;   /* one spacing toward zero */
    }
    uint16_t u; memcpy(&u, &h, 2); return u;
}
"""


def _helper(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / "residual_pairs")
    subprocess.run([gcc, "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
                    "-Wextra", "-Werror", SRC, "-o", exe, "-ldl", "-lpthread"], check=True)
    return gcc, exe


def test_oracle_residual_rounding_equals_binary32_route_on_every_pair(tmp_path):
    _, exe = _helper(tmp_path)
    oracle._load()  # builds liboracle.so if needed
    lib = os.path.join(ROOT, "oracle", "_build", "liboracle.so")
    threads = str(max(1, len(os.sched_getaffinity(0))))
    r = subprocess.run([exe, lib, threads], capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "pairs 4294967296 mismatches 0"


def test_the_pair_check_catches_rounding_toward_zero(tmp_path):
    gcc, exe = _helper(tmp_path)
    src = tmp_path / "truncating.c"
    src.write_text(TRUNCATING)
    so = str(tmp_path / "libtruncating.so")
    subprocess.run([gcc, "-std=c11", "-O2", "-fPIC", "-shared", str(src), "-o", so], check=True)
    r = subprocess.run([exe, so, "2", "4096"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, r.stdout + r.stderr
    assert "first mismatch" in r.stderr
