"""GPU parity of the decoupled-precision Adam step (first moment FP8, second
moment FP16, master weights FP16 with tensor scaling) against the oracle:
bit-exact initial state (fp8_adam_init), first-moment codes, FP16 second
moments and master weights, BF16 weights, amaxes and scales, over several
steps (both sides evaluate the same binary32 operations -- textbook Adam, the
bias corrections as IEEE divisions -- in the same order)."""
import numpy as np
import pytest
import torch

import oracle as o
from helpers import f32_bits

pytestmark = pytest.mark.gpu


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _u16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("n", [16, 4096, 1 << 20, 11008 * 4096 // 64])
@pytest.mark.parametrize("wd,margin", [(0.0, 0), (0.1, 1)])
def test_adam_steps_bit_exact(n, wd, margin):
    f = _lib()
    g = torch.Generator().manual_seed(n + margin)
    w = (torch.randn(n, generator=g) * 0.02).to(torch.bfloat16)
    state = f.Fp8AdamState(w.cuda(), margin=margin)
    hp = f.AdamHyper(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, margin=margin)
    ohp = o.AdamHyper(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, margin=margin)
    # the initial state: fp8_adam_init on the device against the oracle's
    m1, ms, msi, m2, w16, ws, wsi, am = o.adam_init(_u16(w), margin)
    torch.cuda.synchronize()
    assert np.array_equal(state.m1.cpu().numpy(), m1)
    assert np.array_equal(_u16(state.m2), m2)
    assert np.array_equal(_u16(state.w16), w16)
    assert np.array_equal(state.amax.cpu().numpy().view(np.uint32), am.view(np.uint32))
    assert np.array_equal(state.scales.cpu().numpy().view(np.uint32),
                          np.array([ms, msi, ws, wsi], np.float32).view(np.uint32))
    ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws, w_scale_inv=wsi)
    wout = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t in range(1, 5):
        grad = (torch.randn(n, generator=g) * 1e-2 * t).to(torch.bfloat16)
        if t == 3:
            grad[: n // 4] = 0.0
        state.step(grad.cuda(), wout, hp)
        torch.cuda.synchronize()
        m1, ms, msi, m2, w16, ws, wsi, wb, am = o.adam_step(
            _u16(grad), ost["m1"], ost["m1_scale"], ost["m1_scale_inv"], ost["m2"], ost["w16"],
            ost["w_scale"], ost["w_scale_inv"], ohp, t)
        assert np.array_equal(state.m1.cpu().numpy(), m1), t
        assert np.array_equal(_u16(state.m2), m2), t
        assert np.array_equal(_u16(state.w16), w16), t
        assert np.array_equal(_u16(wout), wb), t
        assert np.array_equal(state.amax.cpu().numpy().view(np.uint32), am.view(np.uint32)), t
        gs = state.scales.cpu().numpy()
        assert np.array_equal(gs.view(np.uint32), np.array([ms, msi, ws, wsi], np.float32).view(np.uint32)), t
        ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws,
                   w_scale_inv=wsi)
    f.fp8_sync_status()


def test_adam_full_size_7b_w():
    """Two Adam steps over the full 7B W (11008 x 4096 = 45 M parameters, the
    bench's size and launch): every code of both moments and the master
    weights, the BF16 weights, amaxes and scales against the oracle, bit for
    bit."""
    f = _lib()
    n = 11008 * 4096
    g = torch.Generator().manual_seed(7)
    w = (torch.randn(n, generator=g) * 0.02).to(torch.bfloat16)
    state = f.Fp8AdamState(w.cuda())
    hp = f.AdamHyper(lr=1e-4, weight_decay=0.1)
    ohp = o.AdamHyper(lr=1e-4, weight_decay=0.1)
    m1, ms, msi, m2, w16, ws, wsi, _ = o.adam_init(_u16(w), 0)
    ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws, w_scale_inv=wsi)
    wout = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t in (1, 2):
        grad = (torch.randn(n, generator=g) * 1e-3).to(torch.bfloat16)
        state.step(grad.cuda(), wout, hp)
        torch.cuda.synchronize()
        m1, ms, msi, m2, w16, ws, wsi, wb, am = o.adam_step(
            _u16(grad), ost["m1"], ost["m1_scale"], ost["m1_scale_inv"], ost["m2"], ost["w16"],
            ost["w_scale"], ost["w_scale_inv"], ohp, t)
        assert np.array_equal(state.m1.cpu().numpy(), m1), t
        assert np.array_equal(_u16(state.m2), m2), t
        assert np.array_equal(_u16(state.w16), w16), t
        assert np.array_equal(_u16(wout), wb), t
        assert np.array_equal(state.amax.cpu().numpy().view(np.uint32), am.view(np.uint32)), t
        gs = state.scales.cpu().numpy()
        assert np.array_equal(gs.view(np.uint32),
                              np.array([ms, msi, ws, wsi], np.float32).view(np.uint32)), t
        ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws,
                   w_scale_inv=wsi)
    f.fp8_sync_status()


def test_adam_extreme_gradients():
    """Gradients spread over 1e-30 .. 3e38 with infinities and NaN: second
    moments past FP16's largest value saturate to 65504, first moments and
    weights go non-finite where the pages' arithmetic says so, and NaN
    propagates.  The E4M3 / FP16 state codes, amaxes and scales match the
    oracle bit for bit; the BF16 weight copy too, except that its NaN
    entries are compared as a class (the pages fix no NaN payload: the
    oracle keeps a NaN's sign and payload when it rounds to BF16, the
    kernel's packed conversion writes the canonical NaN), as for the GEMM
    outputs."""
    f = _lib()
    n = 4096 + 16
    g = torch.Generator().manual_seed(99)
    w = (torch.randn(n, generator=g) * 0.02).to(torch.bfloat16)
    state = f.Fp8AdamState(w.cuda())
    hp = f.AdamHyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    ohp = o.AdamHyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    m1, ms, msi, m2, w16, ws, wsi, _ = o.adam_init(_u16(w), 0)
    ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws, w_scale_inv=wsi)
    wout = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t in range(1, 4):
        mag = torch.pow(10.0, torch.empty(n).uniform_(-30, 38.5, generator=g))
        sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
        grad = (mag * sign).to(torch.bfloat16)
        if t >= 2:
            grad[7::997] = float("nan")
            grad[11::1009] = float("inf")
        state.step(grad.cuda(), wout, hp)
        torch.cuda.synchronize()
        m1, ms, msi, m2, w16, ws, wsi, wb, am = o.adam_step(
            _u16(grad), ost["m1"], ost["m1_scale"], ost["m1_scale_inv"], ost["m2"], ost["w16"],
            ost["w_scale"], ost["w_scale_inv"], ohp, t)
        assert np.array_equal(state.m1.cpu().numpy(), m1), t
        assert np.array_equal(_u16(state.m2), m2), t
        assert np.array_equal(_u16(state.w16), w16), t
        got = _u16(wout)
        nan16 = lambda b: (b & 0x7FFF) > 0x7F80
        assert np.array_equal(nan16(got), nan16(wb)), t
        assert np.array_equal(got[~nan16(got)], wb[~nan16(wb)]), t
        assert np.array_equal(state.amax.cpu().numpy().view(np.uint32), am.view(np.uint32)), t
        gs = state.scales.cpu().numpy()
        assert np.array_equal(gs.view(np.uint32),
                              np.array([ms, msi, ws, wsi], np.float32).view(np.uint32)), t
        ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws,
                   w_scale_inv=wsi)
    assert (_u16(state.m2) == 0x7BFF).any()   # saturated second moments occurred
    f.fp8_sync_status()


def test_state_is_five_bytes_per_parameter():
    """First moment 1 B + second moment 2 B + master weights 2 B.  (FP8-LM's
    6 B per parameter also counts an FP8 gradient; this path's gradient, the
    layer's dW, stays BF16.)"""
    f = _lib()
    w = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    s = f.Fp8AdamState(w)
    assert s.m1.element_size() + s.m2.element_size() + s.w16.element_size() == 5


@pytest.mark.parametrize("n", [0, 16, 4096 + 16])
def test_adam_init_edge_cases(n):
    """Empty, one-vector and ragged tensors, all-zero weights (scale 1) and a
    tensor with an infinite weight (scale kept at 1, codes saturate)."""
    f = _lib()
    g = torch.Generator().manual_seed(7 + n)
    cases = [torch.zeros(n, dtype=torch.bfloat16),
             (torch.randn(n, generator=g) * 3.0).to(torch.bfloat16)]
    if n:
        inf = cases[1].clone()
        inf[n // 2] = float("inf")
        cases.append(inf)
    for w in cases:
        st = f.Fp8AdamState(w.cuda(), margin=2)
        torch.cuda.synchronize()
        m1, ms, msi, m2, w16, ws, wsi, am = o.adam_init(_u16(w), 2)
        assert np.array_equal(_u16(st.w16), w16)
        assert np.array_equal(st.m1.cpu().numpy(), m1) and np.array_equal(_u16(st.m2), m2)
        assert np.array_equal(st.scales.cpu().numpy().view(np.uint32),
                              np.array([ms, msi, ws, wsi], np.float32).view(np.uint32))
        assert np.array_equal(st.amax.cpu().numpy().view(np.uint32), am.view(np.uint32))
    f.fp8_sync_status()
