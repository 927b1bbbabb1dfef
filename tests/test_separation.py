"""The oracle and the CUDA path share no code, and the product never runs the
oracle.  Checked on the sources (CPU only)."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "fp8_mixed_precision_amax_gb300")


def _files(d, exts):
    for dp, _, fs in os.walk(d):
        for f in fs:
            if f.endswith(exts):
                yield os.path.join(dp, f)


def test_oracle_does_not_touch_the_package():
    for p in _files(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        src = open(p).read()
        assert "fp8_mixed_precision_amax_gb300" not in src, p
        assert "fp8amax.h" not in src and "csrc" not in src, p


def test_package_does_not_touch_the_oracle():
    pat = re.compile(r"(^|\W)(import\s+oracle|from\s+oracle|oracle/|liboracle|fp8_oracle)")
    for p in _files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        assert not pat.search(open(p).read()), p
    for p in _files(os.path.join(ROOT, "include"), (".h",)):
        assert not pat.search(open(p).read()), p


def test_input_module_holds_no_method_arithmetic():
    src = open(os.path.join(ROOT, "fp8_workloads.py")).read()
    code = "\n".join(l for l in src.splitlines() if not l.strip().startswith("#"))
    body = code.split('"""', 2)[2]  # after the module docstring
    for word in ("float8", "amax(", "448", "57344", "scale_inv", "quantize"):
        assert word not in body, word
