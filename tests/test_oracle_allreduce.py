"""Pins for the oracle's FP8 all-reduce with one shared scale (CPU only).

Source: "Mixed-precision training" wiki note, bullet "per-tensor scaling is
the key": FP8-LM shares one scalar s'_g = min(s'_1, ..., s'_N) across all
GPUs for its FP8 all-reduce.  The sum's definition: the exact sum of the
decoded parts times fl32(1 / s'_g), rounded once to BF16.  Pins: exact
rational arithmetic (fractions.Fraction) with the nearest BF16 found by a
search over the ordered BF16 codes; a worked case where rounding twice would
give another BF16; IEEE non-finite cases; one rank reduces to the plain cast
and dequantisation; the shared scale is the smallest (so no rank's values
saturate); the result approximates the true sum within the FP8 rounding
bound."""
from fractions import Fraction

import numpy as np
import torch

import oracle as o


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


# positive BF16 codes in increasing order of value; 0x7F80 (+inf) stands for
# 2^128, where round-to-nearest overflows
_POS = np.arange(0, 0x7F81, dtype=np.uint32)
_POS_VALS = [Fraction(float(np.uint32(c << 16).view(np.float32))) for c in _POS[:-1]] \
    + [Fraction(2) ** 128]


def nearest_bf16(v: Fraction) -> int:
    """BF16 bits of the exact rational v rounded to nearest, ties to the even
    code, overflowing to infinity; a nonzero v that rounds to 0 keeps its sign."""
    neg = v < 0
    a = -v if neg else v
    lo, hi = 0, len(_POS) - 1
    if a >= _POS_VALS[hi]:
        code = hi
    else:
        while hi - lo > 1:                      # _POS_VALS[lo] <= a < _POS_VALS[hi]
            mid = (lo + hi) // 2
            if _POS_VALS[mid] <= a:
                lo = mid
            else:
                hi = mid
        two_a, mid_v = 2 * a, _POS_VALS[lo] + _POS_VALS[hi]
        code = lo if two_a < mid_v else hi if two_a > mid_v else (lo if lo % 2 == 0 else hi)
    if v == 0:
        return 0
    return int(code) | (0x8000 if neg else 0)


def _exact_sum_bits(parts, fmt, scale):
    table = o.fp8_decode_table(fmt)
    sinv = Fraction(float(np.float32(1.0) / np.float32(scale)))
    out = []
    for col in parts.T:
        out.append(nearest_bf16(sum((Fraction(float(table[c])) for c in col), Fraction(0)) * sinv))
    return np.array(out, np.uint16)


def test_dequant_sum_is_the_exact_sum_rounded_once():
    """Random finite parts of both formats, 1 to 9 ranks, scales that are not
    powers of two (so the product has up to 24 + 48 significant bits), and
    scales whose results land in BF16's subnormal range or overflow it."""
    rng = np.random.default_rng(0)
    for fmt in (o.E4M3, o.E5M2):
        table = o.fp8_decode_table(fmt)
        finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
        for nranks, scale in ((1, 1.0), (2, 37.5), (5, 3.0e-5), (9, 1.7e6), (3, 2.0 ** 120 / 3),
                              (4, 2.0 ** -118 * 0.77)):
            parts = rng.choice(finite, size=(nranks, 400))
            got = o.dequant_sum(parts, fmt, np.float32(scale))
            assert np.array_equal(got, _exact_sum_bits(parts, fmt, np.float32(scale))), \
                (fmt, nranks, scale)


def test_dequant_sum_rounds_once_not_twice():
    """E5M2 parts 57344, 128 and 2^-16 (the smallest subnormal) with scale 1:
    the exact sum 57472 + 2^-16 lies just above the midpoint 57472 of the
    neighbouring BF16 values 57344 and 57600, so the nearest BF16 is 57600
    (0x4761).  Rounding to binary32 first gives exactly 57472, a tie that goes
    to the even 57344 (0x4760)."""
    codes = {v: int(np.nonzero(o.fp8_decode_table(o.E5M2) == v)[0][0])
             for v in (57344.0, 128.0, 2.0 ** -16)}
    parts = np.array([[codes[57344.0]], [codes[128.0]], [codes[2.0 ** -16]]], np.uint8)
    assert o.dequant_sum(parts, o.E5M2, np.float32(1.0))[0] == 0x4761
    # without the smallest part the sum is the midpoint itself: ties to even
    assert o.dequant_sum(parts[:2], o.E5M2, np.float32(1.0))[0] == 0x4760


def test_dequant_sum_non_finite_and_zero_cases():
    e5 = o.E5M2
    pinf, ninf, nan, one, mone = 0x7C, 0xFC, 0x7E, 0x3C, 0xBC   # E5M2 codes
    col = lambda *c: np.array(c, np.uint8).reshape(-1, 1)
    bits = lambda parts, s=1.0: int(o.dequant_sum(parts, e5, np.float32(s))[0])
    is_nan = lambda b: (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0
    assert is_nan(bits(col(one, nan)))
    assert is_nan(bits(col(pinf, ninf, one)))
    assert bits(col(pinf, one, mone)) == 0x7F80
    assert bits(col(ninf, one)) == 0xFF80
    assert bits(col(one, mone)) == 0x0000                        # exact zero: +0
    assert bits(col(0x80, 0x80)) == 0x0000                       # -0 + -0 is an exact zero
    assert bits(col(one), 2.0 ** -130) == 0x7F80                 # 1 / 2^-130 = inf in binary32
    assert bits(col(0x7B), 2.0 ** -120) == 0x7F80                # 1.75 * 2^135 overflows BF16
    assert bits(col(0xFB), 2.0 ** -112) == 0xFF60                # -1.75 * 2^127 is a BF16 value
    # (2 - 2^-8) * 2^127, the midpoint between the largest finite BF16 (an odd
    # code) and 2^128, ties to infinity; 64 * 2^112 below it, the largest finite
    e5_vals = o.fp8_decode_table(o.E5M2)
    mid = col(0x7B, 0x6F, 0x62, 0x58)
    assert e5_vals[mid.ravel()].sum() == 65408.0
    assert bits(mid, 2.0 ** -112) == 0x7F80
    assert bits(np.vstack([mid, col(0xD4)]), 2.0 ** -112) == 0x7F7F
    assert bits(col(0x01), 2.0 ** 125) == 0x0000 | 0x0000       # 2^-16 * 2^-125 = 2^-141 -> +0
    assert bits(col(0x81), 2.0 ** 125) == 0x8000                 # its negative keeps the sign
    assert bits(col(0x01), 2.0 ** 117) == 0x0001                 # 2^-133: the smallest subnormal
    assert is_nan(bits(col(pinf), np.inf))                        # inf * (1 / inf) = inf * 0


def test_one_rank_is_cast_and_dequantise():
    rng = np.random.default_rng(1)
    g = _bf16(rng.standard_normal(4096) * 3e-3)
    out, sg, parts = o.fp8_allreduce([g], o.E5M2)
    assert sg == o.local_scale(g, o.E5M2, 0) == np.float32(57344.0) / o.amax(g)
    table = o.fp8_decode_table(o.E5M2)
    sinv = Fraction(float(np.float32(1.0) / sg))
    ref = np.array([nearest_bf16(Fraction(float(table[c])) * sinv) for c in parts[0]], np.uint16)
    assert np.array_equal(out, ref)
    # an E5M2 value (3 significant bits) times a 24-bit factor is exact in
    # double: torch's BF16 rounding of it agrees wherever binary32 holds it
    dq = table[parts[0]] * np.float64(np.float32(1.0) / sg)
    exact32 = dq.astype(np.float32).astype(np.float64) == dq
    assert np.array_equal(out[exact32], _bf16(dq[exact32].astype(np.float32)))


def test_shared_scale_is_the_minimum_and_sum_is_close():
    rng = np.random.default_rng(2)
    grads = [_bf16(rng.standard_normal(8192) * m) for m in (1e-3, 5e-2, 2e-4, 1e-2)]
    out, sg, parts = o.fp8_allreduce(grads, o.E5M2, margin=0)
    scales = [o.local_scale(g, o.E5M2, 0) for g in grads]
    assert sg == min(scales) and sg == scales[1]          # the largest amax decides
    table = o.fp8_decode_table(o.E5M2)
    assert np.isfinite(table[parts]).all() and (parts & 0x7F).max() == 0x7B
    true = sum(_vals(g) for g in grads)
    mag = sum(np.abs(_vals(g)) for g in grads)
    err = np.abs(_vals(out) - true)
    # each part rounds with relative error <= 2^-3 (E5M2) or, below the
    # normal range, half the smallest subnormal; the sum adds one BF16 rounding
    assert np.all(err <= 2.0 ** -3 * mag + len(grads) * 2.0 ** -17 / sg + 2.0 ** -8 * np.abs(true))
