"""fp8_linear_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (a plugin handed only its input and output tensors by a
framework whose allocator owns the GPU, or code that must not call cudaFree,
which waits for the whole device).  Its FP8 work buffers live in a fixed
array inside the library, so it must give what fp8_linear_bwd gives with
caller-provided buffers, bit for bit (the same deterministic kernels run on
the same bytes), call after call, up to the array's 2^25-element limit.

This file is collected last so that a run stopping at its first failure has
already run every other test.  It also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_workloads as wl
import oracle as o
from helpers import assert_fp8_equal, host_bf16_bits, host_u8


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
    # one element past the limit, either way round
    for M, N in ((4096, 8192 + 16), (4096 + 16, 8192)):
        s = lib.fp8_linear_bwd_noalloc(p16, M, N, 16, ctypes.byref(meta), ctypes.byref(rec),
                                       p16, p16, p16, p16, None)
        assert s == 1 and b"fixed work area" in lib.fp8_last_error()
    # a negative size is fp8_linear_bwd's argument error, not the limit
    s = lib.fp8_linear_bwd_noalloc(p16, -16, 64, 16, ctypes.byref(meta), ctypes.byref(rec),
                                   p16, p16, p16, p16, None)
    assert s != 0 and b"fixed work area" not in lib.fp8_last_error()


def _copy_meta(f, src):
    m = f.Meta(src.history_len)
    m.load_state_dict(src.state_dict())
    return m


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(1040, 784, 400), (4096, 8192, 256)])
def test_noalloc_matches_fp8_linear_bwd_on_two_calls_in_a_row(M, N, K):
    """Two calls in a row, each against fp8_linear_bwd with caller buffers on
    the same inputs and state: dX, dW and every amax slot bit-identical.  The
    caller-buffer call's dY8 / dY8t equal the oracle's cast.  The second
    size fills the array exactly (M * N = 2^25), so the transposed half at
    32 MiB is used to its end.  A warmed second call leaves the device's free
    memory unchanged: the entry point allocates nothing."""
    import fp8_mixed_precision_amax_gb300 as f
    w = wl.Workload("noalloc", M, K, N, "normal", 1.0, 0.05, 1e-2, 16, 0, True, 2)
    W = wl.layer_weight(w, "cuda")
    lin = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    # a few ordinary steps so that the scales are no longer the initial ones
    for step in range(2):
        lin.step(wl.layer_x(w, step, "cuda"), wl.layer_dy(w, step, "cuda"))
    lin.forward(wl.layer_x(w, 2, "cuda"))
    dX_ref = torch.empty((w.M, w.K), dtype=torch.bfloat16, device="cuda")
    dW_ref = torch.empty((w.N, w.K), dtype=torch.bfloat16, device="cuda")
    dX = torch.empty((w.M, w.K), dtype=torch.bfloat16, device="cuda")
    dW = torch.empty((w.N, w.K), dtype=torch.bfloat16, device="cuda")
    free = []
    for call in range(2):
        dY = wl.layer_dy(w, 10 + call, "cuda")
        ma, mb = _copy_meta(f, lin.meta), _copy_meta(f, lin.meta)
        f.fp8_linear_bwd(dY, ma, lin.recipe, lin.X8t, lin.W8t, lin.dY8, lin.dY8t, dX_ref, dW_ref)
        dX.fill_(float("nan"))
        dW.fill_(float("nan"))
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        f.fp8_linear_bwd_noalloc(dY, mb, lin.recipe, lin.X8t, lin.W8t, dX, dW)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        f.fp8_sync_status()
        assert np.array_equal(host_bf16_bits(dX), host_bf16_bits(dX_ref)), f"call {call} dX"
        assert np.array_equal(host_bf16_bits(dW), host_bf16_bits(dW_ref)), f"call {call} dW"
        assert np.array_equal(ma.amax.cpu().numpy().view(np.uint32),
                              mb.amax.cpu().numpy().view(np.uint32)), f"call {call} amax"
        assert mb.amax[f.SLOT_DY].item() > 0 and mb.amax[f.SLOT_DX].item() > 0
        s = np.float32(lin.meta.scale[f.SLOT_DY].item())
        q, qt = o.quantize(host_bf16_bits(dY), s, o.E5M2)
        assert_fp8_equal(host_u8(lin.dY8), q, o.E5M2, f"call {call} dY8")
        assert_fp8_equal(host_u8(lin.dY8t), qt, o.E5M2, f"call {call} dY8t")
    assert free[3] == free[2], free
