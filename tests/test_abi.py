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
    assert lib.fp8_abi_version() == 4


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



def test_host_side_checks_of_the_grouped_layernorm_optimizer_and_reduction_calls():
    """Every argument error below is detected on the host, before any CUDA
    call, with the documented status and a message naming the call."""
    lib = f.library()
    p16 = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1008)
    # bounded-wait self-test: the limit must lie in [1 ns, 5 s]
    for lim in (0, -5, 5_000_000_001):
        s, msg = _err(lib.fp8_selftest_wait_timeout(lim, None))
        assert s == ERR_ARG and "limit_ns" in msg
    # fp32 cast
    assert _err(lib.fp8_quantize_f32(p16, 24, p16, 0, p16, None, None))[0] == ERR_ALIGN
    assert _err(lib.fp8_quantize_f32(p16, 16, p16, 2, p16, None, None))[0] == ERR_ARG
    assert _err(lib.fp8_quantize_f32(odd, 16, p16, 0, p16, None, None))[0] == ERR_ALIGN
    assert _err(lib.fp8_quantize_f32(p16, 16, None, 0, p16, None, None))[0] == ERR_ARG
    # grouped GEMM: one or two problems, each checked like fp8_gemm_tn
    good = api.fp8_gemm_desc(0x1000, 0, 0x1000, 0, 16, 16, 16, 0x1000, 0x1000, 0x1000, None)
    for n in (0, 3):
        s, msg = _err(lib.fp8_gemm_tn_grouped((api.fp8_gemm_desc * 3)(good, good, good), n, None))
        assert s == ERR_ARG and "1 or 2" in msg
    assert _err(lib.fp8_gemm_tn_grouped(None, 1, None))[0] == ERR_ARG
    bad_k = api.fp8_gemm_desc(0x1000, 0, 0x1000, 0, 16, 16, 8, 0x1000, 0x1000, 0x1000, None)
    assert _err(lib.fp8_gemm_tn_grouped((api.fp8_gemm_desc * 2)(good, bad_k), 2, None))[0] \
        == ERR_ALIGN
    bad_f = api.fp8_gemm_desc(0x1000, 5, 0x1000, 0, 16, 16, 16, 0x1000, 0x1000, 0x1000, None)
    assert _err(lib.fp8_gemm_tn_grouped((api.fp8_gemm_desc * 1)(bad_f), 1, None))[0] == ERR_ARG
    # grouped cast
    cd = api.fp8_cast_desc(0x1000, 16, 16, 0x1000, 0x1000, None, None)
    assert _err(lib.fp8_quantize_transpose_grouped((api.fp8_cast_desc * 1)(cd), 0, 0,
                                                   None))[0] == ERR_ARG
    assert _err(lib.fp8_quantize_transpose_grouped((api.fp8_cast_desc * 1)(cd), 1, 9,
                                                   None))[0] == ERR_ARG
    no_out = api.fp8_cast_desc(0x1000, 16, 16, 0x1000, None, None, None)
    s, msg = _err(lib.fp8_quantize_transpose_grouped((api.fp8_cast_desc * 2)(cd, no_out), 2, 0,
                                                     None))
    assert s == ERR_ARG and "both NULL" in msg
    # decode-and-sum of the FP8 all-reduce
    assert _err(lib.fp8_dequant_sum(p16, 0, 16, 1, p16, p16, None))[0] == ERR_ARG
    assert _err(lib.fp8_dequant_sum(p16, 65537, 16, 1, p16, p16, None))[0] == ERR_ARG
    assert _err(lib.fp8_dequant_sum(p16, 2, 16, 3, p16, p16, None))[0] == ERR_ARG
    assert _err(lib.fp8_dequant_sum(p16, 2, 8, 1, p16, p16, None))[0] == ERR_ALIGN
    # Adam on FP8 / FP16 states
    args = [p16, 16, p16, p16, p16, p16, p16, p16, p16, p16, p16]
    assert _err(lib.fp8_adam_step(*args, None, None))[0] == ERR_ARG
    for hp in (api.fp8_adam_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.1, 0.001, 65),
               api.fp8_adam_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.1, 0.001, -1),
               api.fp8_adam_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.0, 0.001, 0),
               api.fp8_adam_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.1, float("nan"), 0)):
        assert _err(lib.fp8_adam_step(*args, ctypes.byref(hp), None))[0] == ERR_ARG
    ok_hp = api.fp8_adam_hyper(1e-3, 0.9, 0.999, 1e-8, 0.0, 0.1, 0.001, 0)
    assert _err(lib.fp8_adam_step(p16, 8, *args[2:], ctypes.byref(ok_hp), None))[0] == ERR_ALIGN
    # LayerNorm + cast
    ln = lambda rows, cols, eps, out, out_t: lib.fp8_layernorm_quantize_transpose(
        p16, p16, p16, rows, cols, eps, p16, 0, out, out_t, None, p16, p16, None)
    s, msg = _err(ln(16, 0, 1e-5, p16, p16))
    assert s == ERR_ARG and "cols" in msg
    assert _err(ln(16, 16, -1.0, p16, p16))[0] == ERR_ARG
    assert _err(ln(16, 16, float("nan"), p16, p16))[0] == ERR_ARG
    assert _err(ln(16, 16, 1e-5, None, None))[0] == ERR_ARG
    assert _err(ln(16, 24, 1e-5, p16, p16))[0] == ERR_ALIGN
    # LayerNorm statistics alone: gamma and beta are needed only with amax
    st = lambda rows, cols, eps, g, am: lib.fp8_layernorm_stats(p16, g, g, rows, cols, eps, p16,
                                                                p16, am, None)
    s, msg = _err(st(16, 0, 1e-5, p16, None))
    assert s == ERR_ARG and "cols" in msg
    assert _err(st(16, 16, -1.0, p16, None))[0] == ERR_ARG
    s, msg = _err(st(16, 16, 1e-5, None, p16))
    assert s == ERR_ARG and "gamma" in msg
    assert _err(st(16, 24, 1e-5, p16, None))[0] == ERR_ALIGN
    assert _err(st(-16, 16, 1e-5, p16, None))[0] == ERR_ARG
    # the allocation-free backward takes at most 2^25 dY elements
    meta = api.fp8_meta(0x1000, 0x1000, 0x1000, 0x1000, 16)
    rec = api.fp8_recipe(0, 16, 1, 0)
    s, msg = _err(lib.fp8_linear_bwd_noalloc(p16, 8192, 8192, 16, ctypes.byref(meta),
                                             ctypes.byref(rec), p16, p16, p16, p16, None))
    assert s == ERR_ARG and "fixed work area" in msg

def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(16, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        f.fp8_amax(x, torch.zeros(1))


def test_header_enums_match_binding():
    """Status codes, formats and scaling modes: the binding's constants are
    the header's enum values."""
    src = open(api.HEADER_PATH).read()
    enum = dict((k, int(v)) for k, v in re.findall(r"\b(FP8_[A-Z0-9_]+)\s*=\s*(\d+)", src))
    assert {v: k for k, v in api.STATUS.items()} == {k: enum[k] for k in api.STATUS.values()}
    assert (enum["FP8_E4M3"], enum["FP8_E5M2"]) == (api.E4M3, api.E5M2)
    assert (enum["FP8_SCALING_DELAYED"], enum["FP8_SCALING_CURRENT"]) == \
        (api.SCALING_DELAYED, api.SCALING_CURRENT)


def test_clock_probe_pointer_must_be_aligned():
    """fp8_set_clock_probe checks its pointer on the host: a misaligned one is
    FP8_ERR_ALIGN; NULL (off) is accepted."""
    from fp8_mixed_precision_amax_gb300 import api
    lib = api.library()
    assert lib.fp8_set_clock_probe(ctypes.c_void_p(0x1004)) == 2
    assert b"8-byte aligned" in lib.fp8_last_error()
    assert lib.fp8_set_clock_probe(None) == 0


def test_layer_logs_its_precision_mode(caplog):
    """A layer logs the precision mode it runs in when it is built (the
    implementation guide's advice to log it at start); building allocates
    buffers only, so CPU tensors serve here."""
    import logging
    import torch
    W = torch.zeros(32, 16, dtype=torch.bfloat16)
    with caplog.at_level(logging.INFO, logger="fp8_mixed_precision_amax_gb300.api"):
        f.Fp8Linear(W, 48, f.Recipe(margin=1, history_len=16, hybrid=True))
        f.Fp8Linear(W, 48, f.Recipe(hybrid=False, current=True))
    msgs = [r.getMessage() for r in caplog.records]
    assert any("[32 x 16]" in m and "E5M2 backward" in m and "delayed" in m and "margin 1" in m
               and "history 16" in m for m in msgs), msgs
    assert any("E4M3 backward" in m and "just-in-time" in m for m in msgs), msgs
