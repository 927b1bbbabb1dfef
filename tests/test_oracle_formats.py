"""Pins for the oracle's FP8 / BF16 codecs (CPU only).

Each check ties the oracle to something other than itself: the numbers the
pages print (tests/golden/fp8_formats.txt), IEEE binary16 (numpy float16, a
textbook routine), torch's CPU float8 / bfloat16 conversions (library
routines), invariants of round-to-nearest-even with saturation, and an
exhaustive run over all 2^32 binary32 patterns against an encoder written
from the formats' bit layouts (tests/exhaustive_encode.c).
"""
import ctypes
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_formats.txt")


def _golden_formats():
    rows = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fmt, e, m, mx, rel, rng = line.split()
        rows[fmt] = dict(e=int(e), m=int(m), max=float(mx), rel=float(rel), rng=rng)
    return rows


FMTS = {"E4M3": o.E4M3, "E5M2": o.E5M2}
TORCH_FP8 = {o.E4M3: torch.float8_e4m3fn, o.E5M2: torch.float8_e5m2}


def test_printed_maxima_and_layouts():
    g = _golden_formats()
    for name, fmt in FMTS.items():
        table = o.fp8_decode_table(fmt)
        finite = table[np.isfinite(table)]
        assert finite.max() == g[name]["max"]
        assert o.fp8_max(fmt) == g[name]["max"]
        # 1 sign + e exponent + m mantissa bits = 8
        assert 1 + g[name]["e"] + g[name]["m"] == 8
        # number of distinct positive normal mantissas is 2^m per binade
        pos = np.unique(finite[finite > 0])
        binade = pos[(pos >= 1.0) & (pos < 2.0)]
        assert len(binade) == 2 ** g[name]["m"]


def test_printed_relative_error_bounds():
    """Worst relative rounding error over the normal range stays within the
    table's ~1e-1 (E4M3) and ~2e-1 (E5M2)."""
    g = _golden_formats()
    worst = {}
    for name, fmt in FMTS.items():
        table = o.fp8_decode_table(fmt)
        pos = np.unique(table[np.isfinite(table) & (table > 0)])
        smallest_normal = 2.0 ** (1 - (2 ** (g[name]["e"] - 1) - 1))
        normal = pos[pos >= smallest_normal]
        # midpoints between neighbours are the worst cases for RNE
        mids = (normal[:-1] + normal[1:]) / 2
        v = np.concatenate([mids * (1 - 2 ** -20), mids * (1 + 2 ** -20)]).astype(np.float32)
        q = o.fp8_encode(v, fmt)
        dq = table[q]
        rel = np.max(np.abs(dq - v.astype(np.float64)) / np.abs(v.astype(np.float64)))
        worst[name] = rel
        assert rel <= g[name]["rel"]
        # worst case sits just above a power of two: u / (1 + u), u = 2^-(m+1)
        u = 2.0 ** -(g[name]["m"] + 1)
        assert rel == pytest.approx(u / (1 + u), rel=1e-3)
    assert worst["E5M2"] == pytest.approx((1 / 9) / (1 / 17) * worst["E4M3"], rel=1e-3)


def test_e5m2_is_top_byte_of_binary16():
    """'Same range as FP16': code c decodes to the binary16 with bits c << 8."""
    table = o.fp8_decode_table(o.E5M2)
    half = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    nan = np.isnan(half)
    assert np.array_equal(np.isnan(table), nan)
    assert np.array_equal(table[~nan], half[~nan])
    g = _golden_formats()
    assert g["E5M2"]["rng"] == "FP16"
    assert np.finfo(np.float16).max == 65504.0 and table[0x7B] == 57344.0


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_decode_matches_torch(fmt):
    table = o.fp8_decode_table(fmt)
    ref = torch.arange(256, dtype=torch.uint8).view(TORCH_FP8[fmt]).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(table), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(table[ok], ref[ok])
    assert np.array_equal(np.signbit(table[ok]), np.signbit(ref[ok]))


def test_e4m3_field_decode_brute_force():
    """Every E4M3 code from its fields: bias 7, subnormals at e == 0, only
    S.1111.111 is NaN (the variant whose maximum is 448)."""
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = o.fp8_decode(c, o.E4M3)
        if e == 15 and m == 7:
            assert math.isnan(v)
            continue
        mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert v == (-mag if s else mag)


def _interesting_f32(fmt, n_random=1 << 21, seed=0):
    """Binary32 values around every FP8 rounding boundary plus random ones,
    all below the point where torch's (non-saturating) cast leaves the format."""
    table = o.fp8_decode_table(fmt)
    pos = np.unique(table[np.isfinite(table) & (table >= 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    pts = np.concatenate([pos, mids]).astype(np.float32)
    bits = pts.view(np.uint32).astype(np.int64)
    around = np.concatenate([bits + d for d in range(-3, 4)])
    around = around[(around >= 0) & (around < 0x7F800000)].astype(np.uint32).view(np.float32)
    rng = np.random.default_rng(seed)
    rb = rng.integers(0, 0x7F800000, n_random, dtype=np.uint32).view(np.float32)
    v = np.concatenate([around, rb])
    limit = 464.0 if fmt == o.E4M3 else 61440.0  # first value torch maps out of range
    v = v[v < limit]
    return np.concatenate([v, -v])


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_encode_matches_torch_in_range(fmt):
    """Round-to-nearest-even against torch's CPU float8 casts, on all values
    where torch's cast does not overflow (torch does not saturate)."""
    v = _interesting_f32(fmt)
    mine = o.fp8_encode(v, fmt)
    ref = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, (v[bad[:5]], mine[bad[:5]], ref[bad[:5]])


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_saturation_and_specials(fmt):
    top = 0x7E if fmt == o.E4M3 else 0x7B
    big = np.array([1e30, np.inf, 3.4e38, o.fp8_max(fmt) * 1.0001, o.fp8_max(fmt) * 1.5],
                   dtype=np.float32)
    assert np.all(o.fp8_encode(big, fmt) == top)
    assert np.all(o.fp8_encode(-big, fmt) == (top | 0x80))
    q = o.fp8_encode(np.array([np.nan, -np.nan], np.float32), fmt)
    assert all(math.isnan(o.fp8_decode(int(c), fmt)) for c in q)
    # signed zero and values below half the smallest subnormal keep their sign
    tiny = np.float32(2.0 ** -40)
    assert list(o.fp8_encode(np.array([0.0, -0.0, tiny, -tiny], np.float32), fmt)) == \
        [0x00, 0x80, 0x00, 0x80]


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_round_trip_monotone_symmetric(fmt):
    table = o.fp8_decode_table(fmt)
    finite = [c for c in range(256) if np.isfinite(table[c])]
    rt = o.fp8_encode(table[finite].astype(np.float32), fmt)
    assert list(rt) == finite
    v = np.sort(np.random.default_rng(1).standard_normal(200000).astype(np.float32) * 300)
    dq = table[o.fp8_encode(v, fmt)]
    assert np.all(np.diff(dq) >= 0)
    q1 = o.fp8_encode(np.abs(v), fmt)
    q2 = o.fp8_encode(-np.abs(v), fmt)
    assert np.array_equal(q2, q1 | 0x80)


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    mine = o.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(mine.view(np.uint32)[~np.isnan(ref)], ref.view(np.uint32)[~np.isnan(ref)])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))


def test_bf16_round_nearest_even_matches_torch():
    rng = np.random.default_rng(2)
    hi = rng.integers(0, 1 << 16, 40000, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    v = (hi[:, None] | lows[None, :]).reshape(-1).view(np.float32)
    mine = o.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(v)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7FFF) > 0x7F80)


def _exhaustive_helper():
    src = os.path.join(os.path.dirname(__file__), "exhaustive_encode.c")
    so = os.path.join(tempfile.mkdtemp(prefix="fp8exh"), "libexhaustive_encode.so")
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-pthread", src, "-o", so],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.count_mismatches.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_uint32)]
    lib.count_mismatches.restype = ctypes.c_int64
    lib.encode_bits_one.argtypes = [ctypes.c_float, ctypes.c_int]
    lib.encode_bits_one.restype = ctypes.c_uint8
    return lib


def test_bit_level_encoder_spot_values():
    """The independent encoder itself on values fixed by the format table:
    the maxima, the smallest subnormals, a tie on each side, saturation."""
    h = _exhaustive_helper()
    cases = {o.E4M3: [(448.0, 0x7E), (464.0, 0x7E), (1e9, 0x7E), (2.0 ** -9, 0x01),
                      (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (1.0625, 0x38),
                      (1.1875, 0x3A), (-2.0, 0xC0), (float("inf"), 0x7E)],
             o.E5M2: [(57344.0, 0x7B), (61440.0, 0x7B), (2.0 ** -16, 0x01), (2.0 ** -17, 0x00),
                      (3 * 2.0 ** -17, 0x02), (1.125, 0x3C), (1.375, 0x3E), (-1.0, 0xBC),
                      (float("-inf"), 0xFB)]}
    for fmt, cs in cases.items():
        for v, code in cs:
            assert h.encode_bits_one(v, fmt) == code, (fmt, v)


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_encode_exhaustive_against_bit_level_encoder(fmt):
    """Every binary32 bit pattern (all 2^32, NaN codes as a class): the
    oracle's nearest-value search over the code table equals an encoder that
    rounds the binary32 significand with integer arithmetic."""
    h = _exhaustive_helper()
    fn = ctypes.cast(o._lib().or_fp8_encode_f32, ctypes.c_void_p)
    first = ctypes.c_uint32(0)
    bad = h.count_mismatches(fn, fmt, max(1, os.cpu_count() or 1), ctypes.byref(first))
    assert bad == 0, (bad, hex(first.value))
