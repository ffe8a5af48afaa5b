"""The product path has no CPU fallback: without the CUDA library the binding
raises, and nothing in the package imports or calls the oracle (which is test
infrastructure only)."""

import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "complex_valued_state_gb300")


def test_missing_library_raises():
    code = ("from complex_valued_state_gb300 import cssd\n"
            "try:\n"
            "    cssd.load('/nonexistent/libcssd.so')\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n"
            "else:\n"
            "    raise SystemExit('no error')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "raised:" in r.stdout and "not built" in r.stdout


def test_package_never_touches_the_oracle():
    pattern = re.compile(r"^\s*(import|from)\s+oracle\b|\boracle\.[A-Za-z_]|liboracle", re.M)
    offenders = []
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                path = os.path.join(dirpath, f)
                with open(path, encoding="utf-8") as fh:
                    if pattern.search(fh.read()):
                        offenders.append(os.path.relpath(path, ROOT))
    assert not offenders, offenders
