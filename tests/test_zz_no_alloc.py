"""fp8_linear_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (a plugin handed only its input and output tensors by a
framework whose allocator owns the GPU, or code that must not call cudaFree,
which waits for the whole device).  Its FP8 work buffers live in a fixed
array inside the library, so it must give what fp8_linear_bwd gives with
caller-provided buffers, call after call.

This file is collected last so that a run stopping at its first failure has
already run every other test.  It also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_workloads as wl
from helpers import assert_gemm_close, host_bf16_bits


def test_noalloc_rejects_sizes_beyond_its_array():
    from fp8_mixed_precision_amax_gb300 import api
    lib = api.library()
    p16 = ctypes.c_void_p(0x1000)
    meta = api.fp8_meta(0x1000, 0x1000, 0x1000, 0x1000, 16)
    rec = api.fp8_recipe(0, 16, 1, 0)
    s = lib.fp8_linear_bwd_noalloc(p16, 8192, 8192, 16, ctypes.byref(meta), ctypes.byref(rec),
                                   p16, p16, p16, p16, None)
    assert s == 1
    assert b"fixed work area" in lib.fp8_last_error()


def _copy_meta(f, src):
    m = f.Meta(src.history_len)
    m.load_state_dict(src.state_dict())
    return m


@pytest.mark.gpu
def test_noalloc_matches_fp8_linear_bwd_on_two_calls_in_a_row():
    import fp8_mixed_precision_amax_gb300 as f
    w = wl.Workload("noalloc", 1040, 400, 784, "normal", 1.0, 0.05, 1e-2, 16, 0, True, 2)
    W = wl.layer_weight(w, "cuda")
    lin = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    # a few ordinary steps so that the scales are no longer the initial ones
    for step in range(2):
        lin.step(wl.layer_x(w, step, "cuda"), wl.layer_dy(w, step, "cuda"))
    lin.forward(wl.layer_x(w, 2, "cuda"))
    for call in range(2):
        dY = wl.layer_dy(w, 10 + call, "cuda")
        ma, mb = _copy_meta(f, lin.meta), _copy_meta(f, lin.meta)
        dX_ref = torch.empty((w.M, w.K), dtype=torch.bfloat16, device="cuda")
        dW_ref = torch.empty((w.N, w.K), dtype=torch.bfloat16, device="cuda")
        f.fp8_linear_bwd(dY, ma, lin.recipe, lin.X8t, lin.W8t, lin.dY8, lin.dY8t, dX_ref, dW_ref)
        dX = torch.full((w.M, w.K), float("nan"), dtype=torch.bfloat16, device="cuda")
        dW = torch.full((w.N, w.K), float("nan"), dtype=torch.bfloat16, device="cuda")
        f.fp8_linear_bwd_noalloc(dY, mb, lin.recipe, lin.X8t, lin.W8t, dX, dW)
        f.fp8_sync_status()
        assert_gemm_close(host_bf16_bits(dX), host_bf16_bits(dX_ref), w.N, f"call {call} dX")
        assert_gemm_close(host_bf16_bits(dW), host_bf16_bits(dW_ref), w.M, f"call {call} dW")
        a, b = ma.amax.cpu().numpy(), mb.amax.cpu().numpy()
        assert a[f.SLOT_DY] == b[f.SLOT_DY] and a[f.SLOT_DY] > 0
        assert abs(float(a[f.SLOT_DX]) - float(b[f.SLOT_DX])) <= 1e-2 * abs(float(a[f.SLOT_DX]))
