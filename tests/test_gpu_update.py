"""GPU parity of the delayed-scaling history / scale update (bit-exact).

Scripted amax sequences (zeros, infinities, denormal amaxes that overflow
the scale, spikes that enter the window, persist L steps and leave) over
history lengths 1 .. 8192, margins 0 .. 3 and both formats.
"""
import numpy as np
import pytest
import torch

import oracle as o

pytestmark = pytest.mark.gpu


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


@pytest.mark.parametrize("L", [1, 16, 512, 1024, 8192])
@pytest.mark.parametrize("margin", [0, 1, 3])
def test_scripted_sequences(L, margin):
    f = _lib()
    T = 6
    mask = 0b101010                       # tensors 1, 3, 5 are E5M2
    fmts = [(mask >> t) & 1 for t in range(T)]
    rng = np.random.default_rng(L * 10 + margin)
    hist = np.zeros((T, L), np.float32)
    scale = np.ones(T, np.float32)
    sinv = np.ones(T, np.float32)
    d_hist = torch.from_numpy(hist).cuda()
    d_amax = torch.zeros(T, device="cuda")
    d_s = torch.ones(T, device="cuda")
    d_si = torch.ones(T, device="cuda")
    steps = 40 if L <= 16 else 12
    for step in range(steps):
        a = np.abs(rng.standard_normal(T) * 10.0 ** rng.integers(-8, 8, T)).astype(np.float32)
        if step % 7 == 3:
            a[step % T] = 0.0
        if step % 11 == 5:
            a[(step + 1) % T] = np.inf
        if step % 9 == 2:
            a[(step + 2) % T] = np.float32(2.0 ** -133)      # scale overflows -> FLT_MAX
        if step == 4:
            a[0] = 1e6                                         # spike
        d_amax.copy_(torch.from_numpy(a))
        f.fp8_scale_update(d_hist, d_amax, d_s, d_si, mask, margin)
        for t in range(T):
            hist[t], scale[t], sinv[t] = o.history_update(hist[t], a[t], scale[t], sinv[t],
                                                          fmts[t], margin)
        torch.cuda.synchronize()
        assert np.array_equal(d_hist.cpu().numpy().view(np.uint32), hist.view(np.uint32)), step
        assert np.array_equal(d_s.cpu().numpy().view(np.uint32), scale.view(np.uint32)), step
        assert np.array_equal(d_si.cpu().numpy().view(np.uint32), sinv.view(np.uint32)), step


def test_layer_update_formats_follow_recipe():
    f = _lib()
    for hybrid in (True, False):
        rc = f.Recipe(margin=0, history_len=8, hybrid=hybrid)
        meta = f.Meta(8)
        meta.amax.copy_(torch.tensor([1.0, 2.0, 4.0, 8.0, 16.0]))
        f.fp8_amax_scale_update(meta, rc)
        torch.cuda.synchronize()
        orc = o.Recipe(margin=0, history_len=8, hybrid=hybrid)
        st = o.State.initial(8)
        st.amax[:] = [1.0, 2.0, 4.0, 8.0, 16.0]
        o.layer_update(st, orc)
        assert np.array_equal(meta.scale.cpu().numpy(), st.scale)
        assert np.array_equal(meta.scale_inv.cpu().numpy(), st.scale_inv)
        assert np.array_equal(meta.history.cpu().numpy(), st.history)
        assert not meta.amax.cpu().numpy().any()       # consumed and cleared
