"""The FP8 Adam step on weights that stress its amax of the new weights,
bit for bit against the oracle (amax, scales, codes, BF16 weights):

* weights whose new values crowd the maximum: all +-0.5 within a few BF16
  steps, with tiny gradients, so that many elements tie or nearly tie;
* weights whose magnitudes grow along the tensor, so that the largest new
  weight sits at the end and every part of the tensor holds a new maximum
  for the elements before it.
"""
import numpy as np
import pytest
import torch

import oracle as o

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _steps_match_oracle(w, grads, lr=3e-3, wd=0.1, margin=0):
    import fp8_mixed_precision_amax_gb300 as f
    n = w.numel()
    state = f.Fp8AdamState(w.cuda(), margin=margin)
    hp = f.AdamHyper(lr=lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, margin=margin)
    ohp = o.AdamHyper(lr=lr, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd, margin=margin)
    m1, ms, msi, m2, w16, ws, wsi, _ = o.adam_init(_u16(w), margin)
    ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws, w_scale_inv=wsi)
    wout = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t, grad in enumerate(grads, start=1):
        state.step(grad.cuda(), wout, hp)
        torch.cuda.synchronize()
        m1, ms, msi, m2, w16, ws, wsi, wb, am = o.adam_step(
            _u16(grad), ost["m1"], ost["m1_scale"], ost["m1_scale_inv"], ost["m2"], ost["w16"],
            ost["w_scale"], ost["w_scale_inv"], ohp, t)
        assert np.array_equal(state.amax.cpu().numpy().view(np.uint32), am.view(np.uint32)), t
        assert np.array_equal(state.scales.cpu().numpy().view(np.uint32),
                              np.array([ms, msi, ws, wsi], np.float32).view(np.uint32)), t
        assert np.array_equal(state.m1.cpu().numpy(), m1), t
        assert np.array_equal(_u16(state.m2), m2), t
        assert np.array_equal(_u16(state.w16), w16), t
        assert np.array_equal(_u16(wout), wb), t
        ost = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws,
                   w_scale_inv=wsi)
    f.fp8_sync_status()


@pytest.mark.parametrize("n", [4096, 1 << 20])
def test_adam_amax_with_weights_crowding_the_maximum(n):
    """All weights +-0.5 (a handful of BF16 neighbours), gradients tiny: the
    new weights differ from the maximum by a few ulps or less."""
    g = torch.Generator().manual_seed(n)
    sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
    jitter = torch.randint(0, 3, (n,), generator=g).float() * 2.0 ** -9
    w = (sign * (0.5 - jitter)).to(torch.bfloat16)
    grads = [(torch.randn(n, generator=g) * 1e-6).to(torch.bfloat16) for _ in range(3)]
    _steps_match_oracle(w, grads)


@pytest.mark.parametrize("n", [4096, 1 << 20])
def test_adam_amax_with_magnitudes_growing_along_the_tensor(n):
    """|w| grows with the index: the maximum is the last element's, and every
    block's elements exceed those of the blocks before it."""
    g = torch.Generator().manual_seed(n + 1)
    mag = torch.linspace(1e-3, 1.0, n)
    sign = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0)
    w = (sign * mag).to(torch.bfloat16)
    grads = [(torch.randn(n, generator=g) * 1e-3).to(torch.bfloat16) for _ in range(3)]
    _steps_match_oracle(w, grads, lr=1e-2)
