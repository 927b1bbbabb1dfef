"""The division by a divisor known in advance that the FP8 Adam step uses for
its bias corrections, m / (1 - b1^t) and v / (1 - b2^t) (the textbook Adam
update, as the oracle divides): q0 = RN(a * RN(1/b)) and two Markstein
corrections.  For each divisor below, every one of the 2^32 binary32 values
of a is divided both ways on the GPU, and the result must equal the IEEE
division bit for bit (NaN as a class).  The divisors are the bias
corrections of the default betas over a range of steps, the ends of the fast
path's range (2^-20 and 1), values just outside it, and log-uniform draws.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def divcheck(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = str(tmp_path_factory.mktemp("divcheck") / "divcheck.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                    "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-o", out,
                    os.path.join(HERE, "cuda", "div_const_check.cu")], check=True)
    lib = ctypes.CDLL(out)
    lib.div_const_check.argtypes = [ctypes.c_float, ctypes.c_int,
                                    ctypes.POINTER(ctypes.c_ulonglong),
                                    ctypes.POINTER(ctypes.c_uint)]
    lib.div_const_one.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.POINTER(ctypes.c_float)]
    return lib


def _divisors():
    bc = set()
    for beta in (0.9, 0.95, 0.99, 0.999, 0.9999):
        for t in (1, 2, 3, 5, 10, 100, 1000, 10000, 100000):
            bc.add(float(np.float32(1.0 - beta ** t)))
    edges = [2.0 ** -20, 2.0 ** -20 * (1 + 2.0 ** -23), 0.5, 0.75, 1.0 - 2.0 ** -24, 1.0,
             float(np.nextafter(np.float32(2.0 ** -20), np.float32(0))), 2.0 ** -24]
    rng = np.random.default_rng(20260)
    draws = [float(np.float32(2.0 ** x)) for x in rng.uniform(-20, 0, 6)]
    return sorted(bc | set(edges) | set(draws))


@pytest.mark.gpu
@pytest.mark.parametrize("b", _divisors())
def test_division_by_known_divisor_is_ieee_for_all_inputs(divcheck, b):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bad, first = ctypes.c_ulonglong(), ctypes.c_uint()
    assert divcheck.div_const_check(b, sms * 8, ctypes.byref(bad), ctypes.byref(first)) == 0
    if bad.value:
        a = np.uint32(first.value).view(np.float32)
        out = (ctypes.c_float * 3)()
        divcheck.div_const_one(float(a), b, out)
        pytest.fail(f"b={b!r}: {bad.value} mismatches; first a={a!r} (0x{first.value:08x}): "
                    f"{out[0]!r} vs IEEE {out[2]!r}")
