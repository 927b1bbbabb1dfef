"""Pins for the oracle's FP8 all-reduce with one shared scale (CPU only).

Source: "Mixed-precision training" wiki note, bullet "per-tensor scaling is
the key": FP8-LM shares one scalar s'_g = min(s'_1, ..., s'_N) across all
GPUs for its FP8 all-reduce.  Pins: the sum against numpy's float64 sum of
the decoded parts; one rank reduces to the plain cast and dequantisation;
the shared scale is the smallest (so no rank's values saturate); the result
approximates the true sum within the FP8 rounding bound."""
import numpy as np
import torch

import oracle as o


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _vals(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def test_dequant_sum_against_numpy():
    rng = np.random.default_rng(0)
    for fmt in (o.E4M3, o.E5M2):
        table = o.fp8_decode_table(fmt)
        finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
        parts = rng.choice(finite, size=(5, 3000))
        s = np.float32(37.5)
        got = _vals(o.dequant_sum(parts, fmt, s))
        exact = table[parts].sum(axis=0) * np.float64(np.float32(1.0) / s)
        ref = _vals(_bf16(exact.astype(np.float32)))
        assert np.array_equal(got, ref)


def test_one_rank_is_cast_and_dequantise():
    rng = np.random.default_rng(1)
    g = _bf16(rng.standard_normal(4096) * 3e-3)
    out, sg, parts = o.fp8_allreduce([g], o.E5M2)
    assert sg == o.local_scale(g, o.E5M2, 0) == np.float32(57344.0) / o.amax(g)
    table = o.fp8_decode_table(o.E5M2)
    ref = _bf16((table[parts[0]] * np.float64(np.float32(1.0) / sg)).astype(np.float32))
    assert np.array_equal(out, ref)


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
