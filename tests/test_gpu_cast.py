"""GPU parity of amax and the fused cast + transpose against the oracle.

Bit-exact: every FP8 byte of both layouts (NaN codes compared as a class) and
the amax word.  Inputs: all 65,536 BF16 bit patterns under many scales,
ragged and multi-tile shapes, planted maxima, and the standalone cast sweep
(2^16 .. 2^28 elements, N(0, 1) with 0.1 % outliers x100) run as amax ->
scale (history of one) -> cast, in E4M3 and E5M2.
"""
import numpy as np
import pytest
import torch

import fp8_workloads as wl
import oracle as o
from helpers import assert_fp8_equal, f32_bits, host_bf16_bits, host_u8

pytestmark = pytest.mark.gpu

FMTS = [o.E4M3, o.E5M2]


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _cast(x, scale, fmt, want_out=True, want_t=True):
    f = _lib()
    rows, cols = x.shape
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    out = torch.full((rows, cols), 0xAA, dtype=torch.uint8, device="cuda") if want_out else None
    out_t = torch.full((cols, rows), 0xAA, dtype=torch.uint8, device="cuda") if want_t else None
    am = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    f.fp8_quantize_transpose(x, s, fmt, out, out_t, am)
    torch.cuda.synchronize()
    return out, out_t, am


def _check(x, scale, fmt, what=""):
    out, out_t, am = _cast(x, scale, fmt)
    xb = host_bf16_bits(x)
    q, qt = o.quantize(xb, np.float32(scale), fmt)
    assert_fp8_equal(host_u8(out), q, fmt, f"{what} out")
    assert_fp8_equal(host_u8(out_t), qt, fmt, f"{what} out_t")
    assert f32_bits(am.cpu().numpy()[0]) == f32_bits(o.amax(xb)), what


ALL_BF16_SCALES = [1.0, 0.5, 3.0, 448.0, 1 / 448.0, 57344.0, 2.0 ** -20, 2.0 ** 20, 1e-30, 1e30,
                   0.0, -1.5, 3.4e38, 1.17549435e-38, 0.1234567, 7.654321e-5, 1234.5678,
                   # degenerate scales the update never produces but the ABI accepts:
                   # IEEE products (inf * x saturates, 0 * inf and NaN give NaN codes)
                   float("inf"), float("-inf"), float("nan"), 1e-45]


@pytest.mark.parametrize("fmt", FMTS)
def test_all_bf16_patterns_under_many_scales(fmt):
    bits = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    rng = np.random.default_rng(100 + fmt)
    scales = ALL_BF16_SCALES + list(np.float32(10.0 ** rng.uniform(-6, 6, 24)))
    for s in scales:
        _check(x, np.float32(s), fmt, f"scale {s}")


@pytest.mark.parametrize("shape", [(16, 16), (48, 80), (128, 128), (144, 272), (256, 4112),
                                   (4224, 16), (1040, 1168)])
@pytest.mark.parametrize("fmt", FMTS)
def test_shapes_ragged_and_multi_tile(shape, fmt):
    g = torch.Generator().manual_seed(shape[0] * 7 + shape[1])
    x = (torch.randn(shape, generator=g) * 30).to(torch.bfloat16).cuda()
    _check(x, np.float32(448.0 / 130.0), fmt, str(shape))


def test_out_only_out_t_only_and_empty():
    f = _lib()
    x = (torch.randn(64, 96) * 5).to(torch.bfloat16).cuda()
    xb = host_bf16_bits(x)
    q, qt = o.quantize(xb, np.float32(2.0), o.E4M3)
    out, _, am = _cast(x, 2.0, o.E4M3, want_t=False)
    assert_fp8_equal(host_u8(out), q, o.E4M3, "out only")
    _, out_t, _ = _cast(x, 2.0, o.E4M3, want_out=False)
    assert_fp8_equal(host_u8(out_t), qt, o.E4M3, "out_t only")
    e = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    am = torch.full((1,), 5.0, device="cuda")
    f.fp8_quantize_transpose(e, torch.ones(1, device="cuda"), 0,
                             torch.empty((0, 32), dtype=torch.uint8, device="cuda"), None, am)
    torch.cuda.synchronize()
    assert am.item() == 0.0


def test_standalone_amax_planted_and_specials():
    f = _lib()
    am = torch.empty(1, device="cuda")
    rng = np.random.default_rng(5)
    for n in [16, 4096, 65536 + 16, 1 << 20]:
        base = rng.standard_normal(n).astype(np.float32)
        for pos in sorted({0, n // 3, n - 1}):
            v = base.copy()
            v[pos] = -777.0
            x = torch.from_numpy(v).to(torch.bfloat16).cuda()
            f.fp8_amax(x, am)
            torch.cuda.synchronize()
            assert f32_bits(am.cpu().numpy()[0]) == f32_bits(o.amax(host_bf16_bits(x)))
    specials = torch.tensor([1.0, float("nan"), -3.0, -0.0] * 4, dtype=torch.bfloat16).cuda()
    f.fp8_amax(specials, am)
    torch.cuda.synchronize()
    assert am.item() == 3.0
    inf = torch.tensor([1.0, float("-inf")] * 8, dtype=torch.bfloat16).cuda()
    f.fp8_amax(inf, am)
    torch.cuda.synchronize()
    assert am.item() == float("inf")
    z = -torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    f.fp8_amax(z, am)
    torch.cuda.synchronize()
    assert f32_bits(am.cpu().numpy()[0]) == 0
    f.fp8_amax(torch.empty(0, dtype=torch.bfloat16, device="cuda"), am)
    torch.cuda.synchronize()
    assert am.item() == 0.0


@pytest.mark.parametrize("n", wl.SWEEP_EXPONENTS)
def test_cast_sweep_amax_scale_cast(n):
    """The standalone quantize sweep: amax, then the scale from a history of
    one (margin 0), then the E4M3 and E5M2 casts with transposed copies.
    Whole tensors are compared up to 2^24 elements; above that, a block of
    rows (and the matching columns of the transposed copy) plus the amax."""
    f = _lib()
    x = wl.sweep_tensor(n, device="cuda")
    rows, cols = x.shape
    xb = host_bf16_bits(x)
    ref_amax = o.amax(xb)
    for fmt in FMTS:
        hist = torch.zeros((1, 1), device="cuda")
        am = torch.empty(1, device="cuda")
        sc = torch.ones(1, device="cuda")
        si = torch.ones(1, device="cuda")
        f.fp8_amax(x, am)
        f.fp8_scale_update(hist, am, sc, si, fmt, 0)
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        am2 = torch.empty(1, device="cuda")
        f.fp8_quantize_transpose(x, sc, fmt, out, out_t, am2)
        torch.cuda.synchronize()
        _, ref_s, ref_si = o.history_update(np.zeros(1, np.float32), ref_amax, 1, 1, fmt, 0)
        assert f32_bits(am.cpu().numpy()[0]) == f32_bits(ref_amax)
        assert f32_bits(am2.cpu().numpy()[0]) == f32_bits(ref_amax)
        assert f32_bits(sc.cpu().numpy()[0]) == f32_bits(ref_s)
        assert f32_bits(si.cpu().numpy()[0]) == f32_bits(ref_si)
        if n <= 24:
            q, qt = o.quantize(xb, ref_s, fmt)
            assert_fp8_equal(host_u8(out), q, fmt, f"2^{n} out")
            assert_fp8_equal(host_u8(out_t), qt, fmt, f"2^{n} out_t")
        else:
            for r0 in (0, rows // 2 + 16, rows - 128):
                blk = xb[r0:r0 + 128]
                q, _ = o.quantize(blk, ref_s, fmt, transpose=False)
                assert_fp8_equal(host_u8(out[r0:r0 + 128]), q, fmt, f"2^{n} rows {r0}")
                assert_fp8_equal(host_u8(out_t[:, r0:r0 + 128]), q.T, fmt, f"2^{n} cols {r0}")
        # the largest element lands on the largest code (margin 0, fresh scale)
        top = 0x7E if fmt == o.E4M3 else 0x7B
        assert int((host_u8(out[: min(rows, 4096)]) & 0x7F).max()) <= top
        del out, out_t


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("margin", [0, 2])
def test_just_in_time_cast(fmt, margin):
    """amax, then the scale from that amax alone, then the cast, in one call:
    bit-exact amax, scale, scale_inv and FP8 bytes; an all-zero tensor keeps
    the previous scale."""
    f = _lib()
    for i, (shape, mag) in enumerate([((128, 128), 1.0), ((144, 272), 3e4), ((1040, 1168), 1e-5),
                                      ((256, 4112), 0.0)]):
        g = torch.Generator().manual_seed(77 + i)
        x = (torch.randn(shape, generator=g) * mag).to(torch.bfloat16).cuda()
        rows, cols = shape
        out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
        am = torch.full((1,), -1.0, device="cuda")
        sc = torch.full((1,), 3.0, device="cuda")
        si = torch.full((1,), 1 / 3.0, device="cuda")
        f.fp8_quantize_transpose_current(x, fmt, margin, am, sc, si, out, out_t)
        torch.cuda.synchronize()
        xb = host_bf16_bits(x)
        ra = o.amax(xb)
        _, rs, rsi = o.history_update(np.zeros(1, np.float32), ra, np.float32(3.0),
                                      np.float32(1 / 3.0), fmt, margin)
        assert f32_bits(am.cpu().numpy()[0]) == f32_bits(ra)
        assert f32_bits(sc.cpu().numpy()[0]) == f32_bits(rs)
        assert f32_bits(si.cpu().numpy()[0]) == f32_bits(rsi)
        q, qt = o.quantize(xb, rs, fmt)
        assert_fp8_equal(host_u8(out), q, fmt, f"{shape}")
        assert_fp8_equal(host_u8(out_t), qt, fmt, f"{shape} t")


@pytest.mark.parametrize("fmt", FMTS)
def test_grouped_cast_of_two_tensors(fmt):
    """Two tensors cast in one launch (as the forward pass casts X and W), each
    with its own scale and amax; also with one of the two empty."""
    f = _lib()
    for shapes in [((1040, 1168), (144, 272)), ((256, 4112), (0, 64))]:
        xs, specs = [], []
        for i, shape in enumerate(shapes):
            g = torch.Generator().manual_seed(300 + i)
            x = (torch.randn(shape, generator=g) * (10.0 ** i)).to(torch.bfloat16).cuda()
            rows, cols = shape
            sc = torch.tensor([np.float32(448.0 / 40.0 / 10.0 ** i)], device="cuda")
            out = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
            out_t = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
            am = torch.full((1,), -1.0, device="cuda")
            xs.append((x, sc, out, out_t, am))
        f.fp8_quantize_transpose_grouped(xs, fmt)
        torch.cuda.synchronize()
        for x, sc, out, out_t, am in xs:
            xb = host_bf16_bits(x)
            q, qt = o.quantize(xb, np.float32(sc.item()), fmt)
            assert_fp8_equal(host_u8(out), q, fmt, "grouped out")
            assert_fp8_equal(host_u8(out_t), qt, fmt, "grouped out_t")
            assert f32_bits(am.cpu().numpy()[0]) == f32_bits(o.amax(xb))


# ------------------------------------------------- fp32 scaled cast (S3) --

def _cast_f32(x: torch.Tensor, scale, fmt):
    f = _lib()
    out = torch.full((x.numel(),), 0xAA, dtype=torch.uint8, device="cuda")
    am = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    f.fp8_quantize_f32(x, torch.tensor([scale], dtype=torch.float32, device="cuda"), fmt, out, am)
    torch.cuda.synchronize()
    return out, am


@pytest.mark.parametrize("fmt", FMTS)
def test_f32_cast_every_binary32_pattern(fmt):
    """All 2^32 binary32 bit patterns, in 16 chunks, cast with scale 1 (so
    fl32(x * 1) = x and the conversion itself is what is compared): every
    code equals the oracle's encoder (NaN codes as a class)."""
    chunk = 1 << 28
    for c in range(16):
        lo = -(1 << 31) + c * chunk
        x = torch.arange(lo, lo + chunk, dtype=torch.int32, device="cuda").view(torch.float32)
        out, _ = _cast_f32(x, np.float32(1.0), fmt)
        ref = o.quantize_f32(np.arange(lo, lo + chunk, dtype=np.int32).view(np.float32),
                             np.float32(1.0), fmt)
        assert_fp8_equal(host_u8(out), ref, fmt, f"chunk {c}")
        del x, out


@pytest.mark.parametrize("n", [16, 4112, (1 << 20) + 48, 3 * (1 << 22)])
@pytest.mark.parametrize("fmt", FMTS)
def test_f32_cast_scaled_with_amax(n, fmt):
    """Scaled casts of fp32 tensors (Gaussian spread over many binades, with
    zeros, infinities, NaN and a planted maximum): codes and amax bit-exact."""
    rng = np.random.default_rng(n + fmt)
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, 6, n)).astype(np.float32)
    k = min(n, 64)
    x[rng.integers(0, n, k)] = np.float32(0.0)
    x[rng.integers(0, n, 2)] = np.float32(np.nan)
    if n > 16:
        x[rng.integers(0, n, 1)] = np.float32(-np.inf)
    x[rng.integers(0, n)] = np.float32(-3.0e7)
    dx = torch.from_numpy(x).cuda()
    for s in (np.float32(1.0), np.float32(1 / 4096.0), np.float32(0.37), np.float32(2.0 ** 20)):
        out, am = _cast_f32(dx, s, fmt)
        assert_fp8_equal(host_u8(out), o.quantize_f32(x, s, fmt), fmt, f"n={n} s={s}")
        assert f32_bits(am.cpu().numpy()[0]) == f32_bits(o.amax_f32(x))


def test_f32_cast_empty_and_argument_checks():
    f = _lib()
    am = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    one = torch.ones(1, device="cuda")
    f.fp8_quantize_f32(torch.empty(0, device="cuda"), one, o.E4M3,
                       torch.empty(0, dtype=torch.uint8, device="cuda"), am)
    torch.cuda.synchronize()
    assert am.item() == 0.0
    with pytest.raises(f.Fp8Error):        # n not a multiple of 16
        f.fp8_quantize_f32(torch.ones(24, device="cuda"), one, o.E4M3,
                           torch.empty(24, dtype=torch.uint8, device="cuda"))
    with pytest.raises(f.Fp8Error):        # bad format
        f.fp8_quantize_f32(torch.ones(32, device="cuda"), one, 7,
                           torch.empty(32, dtype=torch.uint8, device="cuda"))
