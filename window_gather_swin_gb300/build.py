"""Build ``libwgs.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then
one link step produces ``window_gather_swin_gb300/_lib/libwgs.so``.  The
CUDA runtime is linked statically, so the library needs nothing beyond the
driver at load time.

    python -m window_gather_swin_gb300.build [--force] [--verbose] [-DNAME=VALUE ...]
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libwgs.so")

SOURCES = ["wgs_rows.cu", "wgs_gelu.cu", "wgs_gelu_bwd.cu", "wgs_bias_mask.cu", "wgs_runtime.cu",
           "wgs_index.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe:
        return exe
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libwgs.so")


def _inputs_digest(defines) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    h.update(" ".join(ARCH + list(defines)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, defines=(), out: str | None = None) -> str:
    """Compile the library if its sources (or defines) changed; return its path."""
    out = out or LIB
    os.makedirs(os.path.dirname(out), exist_ok=True)
    stamp = out + ".sha256"
    digest = _inputs_digest(defines)
    if not force and os.path.exists(out) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return out
    obj_dir = os.path.join(os.path.dirname(out), "obj")
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "-Xcompiler", "-Wall"] + list(defines)
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, (r.stdout + r.stderr)

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    with open(stamp, "w") as f:
        f.write(digest)
    return out


if __name__ == "__main__":
    args = sys.argv[1:]
    defs = [a for a in args if a.startswith("-D")]
    print(build(force="--force" in args, verbose="--verbose" in args, defines=defs))
