"""The C-ABI library loads, exports every function include/fp8amax.h declares,
and rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import re

import pytest

import fp8_mixed_precision_amax_gb300 as f
from fp8_mixed_precision_amax_gb300 import api

ERR_ARG, ERR_ALIGN = 1, 2


def test_every_declared_function_is_exported():
    lib = f.library()
    declared = f.header_functions()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(lib, name), name
    assert lib.fp8_abi_version() == 3


def test_header_structs_match_binding():
    src = open(api.HEADER_PATH).read()
    meta = re.search(r"typedef struct \{([^}]*)\} fp8_meta;", src).group(1)
    assert [m for m in re.findall(r"(\w+);", meta)] == [n for n, _ in api.fp8_meta._fields_]
    rec = re.search(r"typedef struct \{([^}]*)\} fp8_recipe;", src).group(1)
    assert re.findall(r"(\w+);", rec) == [n for n, _ in api.fp8_recipe._fields_]


def _err(status):
    return status, f.library().fp8_last_error().decode()


def test_host_side_argument_checks():
    lib = f.library()
    p16 = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1008)
    s, msg = _err(lib.fp8_amax(p16, 15, p16, None))
    assert s == ERR_ALIGN and "multiples of 16" in msg
    s, _ = _err(lib.fp8_amax(p16, -16, p16, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_quantize_transpose(p16, 16, 16, p16, 7, p16, None, None, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_quantize_transpose(p16, 16, 16, p16, 0, None, None, None, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_quantize_transpose(odd, 16, 16, p16, 0, p16, None, None, None))
    assert s == ERR_ALIGN
    s, _ = _err(lib.fp8_quantize_transpose(p16, 16, 24, p16, 0, p16, None, None, None))
    assert s == ERR_ALIGN
    s, _ = _err(lib.fp8_gemm_tn(p16, 0, p16, 0, 16, 16, 8, p16, p16, p16, None, None))
    assert s == ERR_ALIGN
    s, _ = _err(lib.fp8_gemm_tn(p16, 0, p16, 3, 16, 16, 16, p16, p16, p16, None, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_gemm_tn(p16, 0, p16, 0, 0, 16, 16, p16, p16, p16, None, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_scale_update(p16, p16, p16, p16, 0, 16, 0, 0, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_scale_update(p16, p16, p16, p16, 5, 16, 0, 65, None))
    assert s == ERR_ARG
    s, _ = _err(lib.fp8_scale_update(p16, p16, p16, p16, 5, 9000, 0, 0, None))
    assert s == ERR_ARG
    meta = api.fp8_meta(0x1000, 0x1000, 0x1000, 0x1000, 16)
    bad = api.fp8_recipe(0, 32, 1, 0)            # history length mismatch
    s, msg = _err(lib.fp8_amax_scale_update(ctypes.byref(meta), ctypes.byref(bad), None))
    assert s == ERR_ARG and "history_len" in msg
    sc = api.fp8_recipe(0, 16, 1, 2)            # neither delayed nor current
    s, msg = _err(lib.fp8_amax_scale_update(ctypes.byref(meta), ctypes.byref(sc), None))
    assert s == ERR_ARG and "scaling" in msg
    s, _ = _err(lib.fp8_quantize_transpose_current(p16, 16, 16, 0, 65, p16, None, p16, p16, p16,
                                                   None))
    assert s == ERR_ARG
    neg = api.fp8_recipe(-1, 16, 1, 0)
    s, _ = _err(lib.fp8_amax_scale_update(ctypes.byref(meta), ctypes.byref(neg), None))
    assert s == ERR_ARG
    ok = api.fp8_recipe(0, 16, 1, 0)
    s, _ = _err(lib.fp8_linear_fwd(p16, p16, 16, 16, 24, ctypes.byref(meta), ctypes.byref(ok),
                                   p16, p16, p16, p16, p16, None))
    assert s == ERR_ALIGN
    s, _ = _err(lib.fp8_linear_bwd(p16, 16, 16, 16, ctypes.byref(meta), ctypes.byref(ok),
                                   p16, None, p16, p16, p16, p16, None))
    assert s == ERR_ARG


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(16, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        f.fp8_amax(x, torch.zeros(1))
