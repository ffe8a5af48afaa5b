"""The source hash behind bench.py's traffic records: comments and whitespace
do not count, code does."""

import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_strip_comments_keeps_literals():
    b = load_bench()
    src = 'a = "x//y /* z */"; // line\nb = \'/\'; /* block\n over lines */ c = 1; d = "\\"//";'
    out = b.strip_comments(src)
    assert '"x//y /* z */"' in out and "'/'" in out and '"\\"//"' in out
    assert "line" not in out and "block" not in out and "over lines" not in out


def test_code_changes_and_only_code_changes_count():
    b = load_bench()
    base = "int f(int x) {\n    return x + 1;  // add one\n}\n"

    def h(s):
        return " ".join(b.strip_comments(s).split())

    assert h(base) == h("// a new header\n// of two lines\nint f(int x) {\n  return x + 1;\n}\n")
    assert h(base) == h("int f(int x) { /* inline */ return x + 1; }")
    assert h(base) != h("int f(int x) {\n    return x + 2;  // add one\n}\n")
