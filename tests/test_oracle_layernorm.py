"""Pins for the oracle's LayerNorm (CPU only): torch's float64 layer_norm (a
library routine) and the normalisation invariants (zero mean, unit variance
before the affine part)."""
import numpy as np
import torch

import oracle as o


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def test_layernorm_matches_torch_float64():
    rng = np.random.default_rng(0)
    for rows, cols in [(1, 16), (7, 48), (64, 4096), (3, 8192)]:
        x = _bf16(rng.standard_normal((rows, cols)) * 3 + 1.5)
        g = _bf16(rng.standard_normal(cols))
        b = _bf16(rng.standard_normal(cols) * 0.1)
        y, mean, rstd = o.layernorm(x, g, b, 1e-5)
        ref = torch.nn.functional.layer_norm(_f64(x), (cols,), _f64(g), _f64(b), eps=1e-5).numpy()
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        xd = _f64(x).numpy()
        assert np.allclose(mean, xd.mean(axis=1), rtol=1e-13, atol=1e-13)
        assert np.allclose(rstd, 1 / np.sqrt(xd.var(axis=1) + 1e-5), rtol=1e-12)


def test_layernorm_normalises_rows():
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((32, 1024)) * 100 - 7)
    ones, zeros = _bf16(np.ones(1024)), _bf16(np.zeros(1024))
    y, _, _ = o.layernorm(x, ones, zeros, 0.0)
    assert np.allclose(y.mean(axis=1), 0, atol=1e-12)
    assert np.allclose(y.var(axis=1), 1, rtol=1e-12)
    # gamma scales and beta shifts each column
    g = _bf16(np.full(1024, 2.0))
    b = _bf16(np.full(1024, 0.5))
    y2, _, _ = o.layernorm(x, g, b, 0.0)
    assert np.allclose(y2, 2 * y + 0.5, rtol=1e-14, atol=1e-14)


def test_layernorm_closed_forms():
    """Rows whose statistics are known exactly: a constant row has mean c,
    variance 0, rstd 1/sqrt(eps) and output beta; a row alternating a and b
    has mean (a+b)/2 and variance ((a-b)/2)^2, so its normalised values are
    +-1 scaled by sqrt(var / (var + eps))."""
    cols = 256
    g = _bf16(np.full(cols, 1.5))
    b = _bf16(np.linspace(-1, 1, cols))
    x = _bf16(np.full((1, cols), 3.25))
    y, mean, rstd = o.layernorm(x, g, b, 1e-5)
    assert mean[0] == 3.25 and rstd[0] == 1 / np.sqrt(1e-5)
    assert np.array_equal(y[0], _f64(b).numpy())
    a_, b_ = 2.0, -6.0
    x = _bf16(np.tile([a_, b_], cols // 2)[None, :])
    y, mean, rstd = o.layernorm(x, _bf16(np.ones(cols)), _bf16(np.zeros(cols)), 1e-5)
    var = ((a_ - b_) / 2) ** 2
    assert mean[0] == (a_ + b_) / 2
    assert np.isclose(rstd[0], 1 / np.sqrt(var + 1e-5), rtol=1e-15)
    expect = np.tile([1.0, -1.0], cols // 2) * np.sqrt(var) / np.sqrt(var + 1e-5)
    assert np.allclose(y[0], expect, rtol=1e-14, atol=0)
