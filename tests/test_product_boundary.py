"""The product path and the oracle stay apart, and the product has no CPU path.

The oracle is test infrastructure: the package (its Python binding and its
CUDA / C++ sources) must never import, include or call it, the two must share
no code, and a missing library must raise rather than fall back to anything.
"""
import ast
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "window_gather_swin_gb300")
CSRC = os.path.join(PKG, "csrc")
ORACLE = os.path.join(ROOT, "oracle")


def _py_files(d):
    for base, _, files in os.walk(d):
        if "__pycache__" in base or "_lib" in base:
            continue
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(base, f)


def _imported_modules(path):
    tree = ast.parse(open(path).read(), path)
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            yield from (a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.module:
            yield node.module


def test_package_never_imports_the_oracle():
    for path in _py_files(PKG):
        for mod in _imported_modules(path):
            assert mod.split(".")[0] != "oracle", f"{path} imports {mod}"


def test_library_sources_never_reach_the_oracle():
    for name in os.listdir(CSRC):
        text = open(os.path.join(CSRC, name)).read()
        assert not re.search(r"#\s*include\s*[<\"][^>\"]*oracle", text), name
        assert not re.search(r"\borc_\w+\s*\(", text), f"{name} calls an oracle function"


def test_oracle_shares_no_code_with_the_library():
    for name in os.listdir(ORACLE):
        if not name.endswith((".c", ".h", ".py")):
            continue
        text = open(os.path.join(ORACLE, name)).read()
        assert "wgs.h" not in text and "csrc" not in text, name
    for path in _py_files(ORACLE):
        for mod in _imported_modules(path):
            assert mod.split(".")[0] != "window_gather_swin_gb300", f"{path} imports {mod}"


def test_missing_library_raises_instead_of_falling_back():
    """With no library and no way to build one, loading raises."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from window_gather_swin_gb300 import _capi, build\n"
        "def fail(*a, **k): raise RuntimeError('no toolkit')\n"
        "build.build = fail\n"
        "try:\n"
        "    _capi.load('/nonexistent/libwgs.so')\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "else:\n"
        "    print('loaded')\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised:" in r.stdout and "not built" in r.stdout, r.stdout
