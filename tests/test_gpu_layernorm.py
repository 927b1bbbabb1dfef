"""GPU parity of LayerNorm fused with the scaled cast (te.LayerNorm in front of
an FP8 linear) against the oracle's double-precision LayerNorm.

The statistics are fp32 sums on the GPU and exact sums in the oracle, so y
agrees to a few fp32 rounding errors of the terms it combines, not bit for
bit.  Hence: mean / rstd / amax(y) within 1e-5 relative; every FP8 code is a
correct cast of some value within that error band around the oracle's exact
y * s (band = 2^-16 x ((|x| + |mean|) * rstd * |gamma| + |beta|) * s), and
codes that differ from the cast of the exact value must be rare.

The elementwise part is checked bit for bit on its own: given the kernel's
own mean and rstd, y = ((x - mean) * rstd) * gamma + beta evaluated in numpy
float32 (one rounding per operation, nothing fused), times s and cast by the
oracle's encoder, must reproduce every code and the amax exactly."""
import numpy as np
import pytest
import torch

import fp8_workloads as wl
import oracle as o
from helpers import assert_codes_in_band, assert_gemm_close, bf16_values, host_bf16_bits, host_u8

pytestmark = pytest.mark.gpu
REL = 2.0 ** -16


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _inputs(rows, cols, seed, mag=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, cols, generator=g) * mag * 3 + mag).to(torch.bfloat16)
    gamma = (1 + 0.2 * torch.randn(cols, generator=g)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(cols, generator=g)).to(torch.bfloat16)
    return x.cuda(), gamma.cuda(), beta.cuda()


def check_elementwise_exact(gpu, x, gamma, beta, mean_gpu, rstd_gpu, s, fmt, amax_gpu, what):
    """x, gamma, beta as BF16 bits; mean_gpu, rstd_gpu the kernel's fp32 statistics."""
    widen = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)
    xf = widen(x)
    mu = np.asarray(mean_gpu, np.float32)[:, None]
    rs = np.asarray(rstd_gpu, np.float32)[:, None]
    y = (((xf - mu) * rs) * widen(gamma)[None, :]) + widen(beta)[None, :]
    assert y.dtype == np.float32
    ref = o.fp8_encode((y * np.float32(s)).astype(np.float32), fmt).reshape(y.shape)
    from helpers import assert_fp8_equal
    assert_fp8_equal(gpu, ref, fmt, what + " (elementwise, bit-exact)")
    if amax_gpu is not None:
        a = np.abs(y)
        assert np.float32(amax_gpu).view(np.uint32) == np.float32(a[~np.isnan(a)].max()).view(np.uint32)


def check_codes(gpu, x, gamma, beta, mean, rstd, y, s, fmt, what):
    """x, gamma, beta as BF16 bits; mean, rstd, y from the oracle (double)."""
    xd = bf16_values(x)
    mag = (np.abs(xd) + np.abs(mean)[:, None]) * rstd[:, None] * np.abs(bf16_values(gamma)) + \
        np.abs(bf16_values(beta))
    return assert_codes_in_band(gpu, y * np.float64(s), REL * mag * np.float64(s), fmt, what)


@pytest.mark.parametrize("rows,cols", [(16, 16), (144, 272), (1040, 4096), (256, 8192),
                                       (48, 12288)])
@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_layernorm_cast_matches_oracle(rows, cols, fmt):
    f = _lib()
    x, gamma, beta = _inputs(rows, cols, rows + cols + fmt)
    s = np.float32(448.0 / 6.0) if fmt == o.E4M3 else np.float32(57344.0 / 6.0)
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    am = torch.full((1,), -1.0, device="cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    f.fp8_layernorm_quantize_transpose(x, gamma, beta, 1e-5, torch.tensor([s], device="cuda"),
                                       fmt, mean, rstd, out, out_t, am)
    torch.cuda.synchronize()
    xb, gb, bb = host_bf16_bits(x), host_bf16_bits(gamma), host_bf16_bits(beta)
    y, mu, rs = o.layernorm(xb, gb, bb, 1e-5)
    assert np.allclose(mean.cpu().numpy(), mu, rtol=1e-5, atol=1e-5 * np.abs(mu).max())
    assert np.allclose(rstd.cpu().numpy(), rs, rtol=1e-5)
    assert abs(am.item() - np.abs(y).max()) <= 1e-5 * np.abs(y).max()
    q = host_u8(out)
    check_codes(q, xb, gb, bb, mu, rs, y, s, fmt, f"{rows}x{cols} out")
    check_elementwise_exact(q, xb, gb, bb, mean.cpu().numpy(), rstd.cpu().numpy(), s, fmt,
                            am.item(), f"{rows}x{cols}")
    assert np.array_equal(host_u8(out_t), q.T)


@pytest.mark.parametrize("M,K,N", [(1040, 1024, 784), (272, 4112, 144)])
def test_layernorm_linear_step_matches_oracle(M, K, N):
    """One step of LayerNorm + FP8 linear (te.LayerNormLinear) then the
    linear's backward, against the oracle: LN(X) codes as above, Y / dX / dW
    within the GEMM tolerance; a second step under just-in-time scaling.
    K = 1024 takes the one-pass LayerNorm cast under delayed scaling, K = 4112
    (past its 4096-column limit) the statistics kernel and the cast kernel's
    LayerNorm branch."""
    f = _lib()
    w = wl.Workload("ln", M, K, N, "normal", 1.0, 0.03, 1e-2, 16, 0, True, 2)
    W = wl.layer_weight(w, "cuda")
    for current in (False, True):
        _, gamma, beta = _inputs(16, w.K, 5)
        lin = f.Fp8LayerNormLinear(W, w.M, gamma, beta, 1e-5,
                                   f.Recipe(w.margin, w.history_len, w.hybrid, current=current))
        X, dY = wl.layer_x(w, 0, "cuda"), wl.layer_dy(w, 0, "cuda")
        lin.forward(X)
        lin.backward(dY)
        torch.cuda.synchronize()
        xb, gb, bb = host_bf16_bits(X), host_bf16_bits(gamma), host_bf16_bits(beta)
        y, mu, rs = o.layernorm(xb, gb, bb, 1e-5)
        sx = np.float32(448.0 / np.abs(y).max()) if current else np.float32(1.0)
        assert abs(lin.meta.scale[o.SLOT_X].item() - sx) <= 1e-5 * sx
        assert abs(lin.meta.amax[o.SLOT_X].item() - np.abs(y).max()) <= 1e-5 * np.abs(y).max()
        X8 = host_u8(lin.X8)
        assert np.array_equal(host_u8(lin.X8t), X8.T)
        check_codes(X8, xb, gb, bb, mu, rs, y, lin.meta.scale[o.SLOT_X].item(), o.E4M3,
                    "LN(X) codes")
        check_elementwise_exact(X8, xb, gb, bb, lin.mean.cpu().numpy(), lin.rstd.cpu().numpy(),
                                lin.meta.scale[o.SLOT_X].item(), o.E4M3, None, "LN(X)")
        # the GEMMs from the GPU's own FP8 operands (parity of the GEMM itself is
        # tested elsewhere); the operands must be the oracle's up to tie codes
        rc = o.Recipe(w.margin, w.history_len, w.hybrid)
        fm = rc.formats()
        W8, W8t = o.quantize(host_bf16_bits(W), np.float32(lin.meta.scale[o.SLOT_W].item()), fm[1])
        assert np.array_equal(host_u8(lin.W8), W8)
        si = lin.meta.scale_inv.cpu().numpy()
        ref = o.epilogue(o.gemm_tn(X8, fm[0], W8, fm[1]), si[0], si[1])
        assert_gemm_close(host_bf16_bits(lin.Y), ref, w.K, "Y")
        dY8, dY8t = o.quantize(host_bf16_bits(dY), np.float32(lin.meta.scale[o.SLOT_DY].item()),
                               fm[3])
        ref = o.epilogue(o.gemm_tn(dY8t, fm[3], X8.T.copy(), fm[0]), si[3], si[0])
        assert_gemm_close(host_bf16_bits(lin.dW), ref, w.M, "dW")
    f.fp8_sync_status()


def _ln_cast(f, x, gamma, beta, s, fmt, row_major, transposed):
    rows, cols = x.shape
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda") if row_major else None
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda") if transposed else None
    am = torch.full((1,), -1.0, device="cuda")
    mean = torch.full((rows,), float("nan"), device="cuda")
    rstd = torch.full((rows,), float("nan"), device="cuda")
    f.fp8_layernorm_quantize_transpose(x, gamma, beta, 1e-5, torch.tensor([s], device="cuda"),
                                       fmt, mean, rstd, out, out_t, am)
    f.fp8_sync_status()
    bits = lambda t: t.cpu().numpy().view(np.uint32)
    return (host_u8(out) if row_major else None), (host_u8(out_t) if transposed else None), \
        bits(mean), bits(rstd), bits(am)[0]


@pytest.mark.parametrize("rows,cols", [(16, 16), (48, 272), (1040, 1024), (1040, 4096),
                                       (8192, 4096), (48, 4112), (144, 400), (6080, 400)])
@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_layernorm_cast_one_pass_matches_two_kernels(rows, cols, fmt):
    """Rows of up to 4096 columns with a row-major output take the one-pass
    kernel (statistics, normalisation and cast from one read of x), and the
    transposed copy, when asked for, is the byte transpose of its codes.
    Three calls on the same input: row-major only, both outputs, transposed
    only (this last one takes the two-kernel path: statistics kernel, then the
    cast with its transposed copy).  Codes, mean, rstd and amax agree bit for
    bit across all three, up to the 7B layer's X (8192 x 4096), and the
    result is checked against the oracle as above.  (48, 4112) is past the
    one-pass limit and takes two kernels every time; (144, 400) has ragged
    128 x 128 transpose tiles; (6080, 400) gives each CTA 40 rows over its 32
    row buffers, so the warps owning two buffers take rows from both."""
    f = _lib()
    x, gamma, beta = _inputs(rows, cols, 77 + rows + fmt)
    s = np.float32(448.0 / 6.0) if fmt == o.E4M3 else np.float32(57344.0 / 6.0)
    q1, _, m1, r1, a1 = _ln_cast(f, x, gamma, beta, s, fmt, True, False)
    q2, q2t, m2, r2, a2 = _ln_cast(f, x, gamma, beta, s, fmt, True, True)
    _, q3t, m3, r3, a3 = _ln_cast(f, x, gamma, beta, s, fmt, False, True)
    assert np.array_equal(m1, m2) and np.array_equal(r1, r2) and a1 == a2
    assert np.array_equal(m1, m3) and np.array_equal(r1, r3) and a1 == a3
    assert np.array_equal(q1, q2)
    assert np.array_equal(q2t, q1.T)
    assert np.array_equal(q3t, q1.T)
    xb, gb, bb = host_bf16_bits(x), host_bf16_bits(gamma), host_bf16_bits(beta)
    y, mu, rs = o.layernorm(xb, gb, bb, 1e-5)
    mean = m2.view(np.float32)
    assert np.allclose(mean, mu, rtol=1e-5, atol=1e-5 * np.abs(mu).max())
    assert np.allclose(r2.view(np.float32), rs, rtol=1e-5)
    check_elementwise_exact(q2, xb, gb, bb, mean, r2.view(np.float32), s, fmt,
                            np.uint32(a2).view(np.float32), f"{rows}x{cols}")


def _random_shapes(n, seed):
    rng = np.random.default_rng(seed)
    return [(16 * int(rng.integers(1, 190)), 16 * int(rng.integers(1, 257))) for _ in range(n)]


@pytest.mark.parametrize("rows,cols", _random_shapes(12, 4242))
def test_layernorm_cast_random_shapes(rows, cols):
    """Seeded random shapes (multiples of 16 up to 3024 x 4096, mostly not of
    128: ragged transpose tiles and uneven rows per CTA): the one-pass cast,
    its byte transpose and the two-kernel path agree bit for bit, and the
    codes are exact given the kernels' statistics."""
    f = _lib()
    x, gamma, beta = _inputs(rows, cols, rows * 7 + cols)
    s = np.float32(448.0 / 6.0)
    q1, _, m1, r1, a1 = _ln_cast(f, x, gamma, beta, s, o.E4M3, True, False)
    q2, q2t, m2, r2, a2 = _ln_cast(f, x, gamma, beta, s, o.E4M3, True, True)
    _, q3t, m3, r3, a3 = _ln_cast(f, x, gamma, beta, s, o.E4M3, False, True)
    assert np.array_equal(q1, q2) and np.array_equal(q2t, q1.T) and np.array_equal(q3t, q1.T)
    assert np.array_equal(m1, m2) and np.array_equal(m1, m3)
    assert np.array_equal(r1, r2) and np.array_equal(r1, r3) and a1 == a2 == a3
    xb, gb, bb = host_bf16_bits(x), host_bf16_bits(gamma), host_bf16_bits(beta)
    check_elementwise_exact(q1, xb, gb, bb, m1.view(np.float32), r1.view(np.float32), s, o.E4M3,
                            np.uint32(a1).view(np.float32), f"{rows}x{cols}")


@pytest.mark.parametrize("rows,cols", [(16, 16), (1040, 4096), (6080, 400), (256, 8192),
                                       (48, 12288)])
def test_layernorm_stats_alone(rows, cols):
    """fp8_layernorm_stats gives the mean, rstd and max |y| of the LayerNorm
    cast bit for bit (the register, shared-memory and looping statistics
    kernels), and without amax needs neither gamma nor beta."""
    f = _lib()
    x, gamma, beta = _inputs(rows, cols, 5 + rows + cols)
    s = np.float32(448.0 / 6.0)
    q, _, m_ref, r_ref, a_ref = _ln_cast(f, x, gamma, beta, s, o.E4M3, True, False)
    mean = torch.full((rows,), float("nan"), device="cuda")
    rstd = torch.full((rows,), float("nan"), device="cuda")
    am = torch.full((1,), -1.0, device="cuda")
    f.fp8_layernorm_stats(x, gamma, beta, 1e-5, mean, rstd, am)
    f.fp8_sync_status()
    bits = lambda t: t.cpu().numpy().view(np.uint32)
    assert np.array_equal(bits(mean), m_ref) and np.array_equal(bits(rstd), r_ref)
    assert bits(am)[0] == a_ref
    mean.fill_(float("nan"))
    rstd.fill_(float("nan"))
    f.fp8_layernorm_stats(x, None, None, 1e-5, mean, rstd)
    f.fp8_sync_status()
    assert np.array_equal(bits(mean), m_ref) and np.array_equal(bits(rstd), r_ref)
    # and against the oracle's fp64 statistics
    _, mu, rs = o.layernorm(host_bf16_bits(x), host_bf16_bits(gamma), host_bf16_bits(beta), 1e-5)
    assert np.allclose(m_ref.view(np.float32), mu, rtol=1e-5, atol=1e-5 * np.abs(mu).max())
    assert np.allclose(r_ref.view(np.float32), rs, rtol=1e-5)


def test_layernorm_stats_no_rows():
    """No rows: nothing is read, and amax is overwritten with 0."""
    f = _lib()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    am = torch.full((1,), -1.0, device="cuda")
    e = torch.empty(0, device="cuda")
    f.fp8_layernorm_stats(x, g, g, 1e-5, e, e, am)
    f.fp8_sync_status()
    assert am.item() == 0.0


@pytest.mark.parametrize("cols", [4096, 8192, 12288])
def test_layernorm_constant_rows(cols):
    """Degenerate rows whose elements are all equal: the variance is 0, so
    rstd = 1/sqrt(eps) and the output is beta exactly.  At power-of-two
    widths the fp32 mean is exact and those closed forms are checked bit for
    bit; at every width (the register and the looping statistics kernels)
    the elementwise result is exact given the kernel's own statistics."""
    f = _lib()
    rows = 32
    x = torch.full((rows, cols), 3.25, dtype=torch.bfloat16, device="cuda")
    x[1::2] = -0.5
    g = torch.Generator().manual_seed(cols)
    gamma = (1 + 0.2 * torch.randn(cols, generator=g)).to(torch.bfloat16).cuda()
    beta = (0.1 * torch.randn(cols, generator=g)).to(torch.bfloat16).cuda()
    s = np.float32(64.0)
    out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    am = torch.full((1,), -1.0, device="cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    f.fp8_layernorm_quantize_transpose(x, gamma, beta, 1e-5, torch.tensor([s], device="cuda"),
                                       o.E4M3, mean, rstd, out, out_t, am)
    torch.cuda.synchronize()
    xb, gb, bb = host_bf16_bits(x), host_bf16_bits(gamma), host_bf16_bits(beta)
    q = host_u8(out)
    check_elementwise_exact(q, xb, gb, bb, mean.cpu().numpy(), rstd.cpu().numpy(), s, o.E4M3,
                            am.item(), f"constant rows x {cols}")
    assert np.array_equal(host_u8(out_t), q.T)
    if cols & (cols - 1) == 0:
        m = mean.cpu().numpy()
        assert np.all(m[0::2] == np.float32(3.25)) and np.all(m[1::2] == np.float32(-0.5))
        rs = np.float32(np.float32(1.0) / np.sqrt(np.float32(1e-5)))
        assert np.all(rstd.cpu().numpy().view(np.uint32) == rs.view(np.uint32))
        ref, _ = o.quantize(np.tile(bb, (rows, 1)), s, o.E4M3)
        assert np.array_equal(q, ref)
