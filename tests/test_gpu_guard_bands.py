"""Out-of-range writes: every output is allocated with a guard band of
sentinel bytes after it (and the buffer itself pre-filled with a canary), on
ragged shapes; after the call the guard band must be untouched.  This is the
stray-write half of what a memory checker would report (the canary checks in
the parity tests cover missed writes)."""
import numpy as np
import pytest
import torch

import oracle as o

pytestmark = pytest.mark.gpu
GUARD = 4096


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _guarded(n, dtype):
    """A view of n elements at the start of a buffer followed by GUARD bytes of 0xA5."""
    esize = torch.empty(0, dtype=dtype).element_size()
    raw = torch.full((n * esize + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    return raw, raw[: n * esize].view(dtype)


def _intact(raw, n_bytes):
    tail = raw[n_bytes:].cpu().numpy()
    return bool(np.all(tail == 0xA5))


@pytest.mark.parametrize("rows,cols", [(16, 48), (144, 272), (400, 1040), (1040, 784)])
@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_cast_outputs_stay_in_bounds(rows, cols, fmt):
    f = _lib()
    x = torch.randn(rows, cols, device="cuda").to(torch.bfloat16)
    ro, out = _guarded(rows * cols, torch.uint8)
    rt, out_t = _guarded(rows * cols, torch.uint8)
    ra, am = _guarded(1, torch.float32)
    f.fp8_quantize_transpose(x, torch.ones(1, device="cuda"), fmt, out.view(rows, cols),
                             out_t.view(cols, rows), am)
    torch.cuda.synchronize()
    assert _intact(ro, rows * cols) and _intact(rt, rows * cols) and _intact(ra, 4)


@pytest.mark.parametrize("M,N,K", [(16, 16, 16), (144, 272, 48), (400, 784, 1040), (1040, 400, 128)])
def test_gemm_output_stays_in_bounds(M, N, K):
    f = _lib()
    A = torch.randint(0, 0x7E, (M, K), dtype=torch.uint8, device="cuda")
    B = torch.randint(0, 0x7E, (N, K), dtype=torch.uint8, device="cuda")
    rd, D = _guarded(M * N, torch.bfloat16)
    ra, am = _guarded(1, torch.float32)
    one = torch.ones(1, device="cuda")
    f.fp8_gemm_tn(A, o.E4M3, B, o.E4M3, one, one, D.view(M, N), am)
    torch.cuda.synchronize()
    assert _intact(rd, 2 * M * N) and _intact(ra, 4)


def test_fp32_cast_and_sum_stay_in_bounds():
    f = _lib()
    n = 4112
    x = torch.randn(n, device="cuda")
    ro, out = _guarded(n, torch.uint8)
    f.fp8_quantize_f32(x, torch.ones(1, device="cuda"), o.E4M3, out)
    parts = torch.randint(0, 0x7B, (3, n), dtype=torch.uint8, device="cuda")
    rs, s = _guarded(n, torch.bfloat16)
    f.fp8_dequant_sum(parts, o.E5M2, torch.ones(1, device="cuda"), s)
    torch.cuda.synchronize()
    assert _intact(ro, n) and _intact(rs, 2 * n)
