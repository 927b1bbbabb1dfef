"""Pins for the oracle's FP8 GEMM, dequant epilogue and layer step (CPU only).

Sources: "Mixed-precision training" wiki note, bullet "extension to FP8" (only
the GEMMs run in FP8, accumulation in higher precision); te.Linear forward and
backward under fp8_autocast with Format.HYBRID ("NVIDIA Transformer Engine and
FP8 mixed precision: implementation guide", sections "Basic structure of FP8
training code" and "Dynamic scaling and the FP8 recipe").

Pins: exact rational arithmetic (fractions.Fraction) on tiny shapes, numpy's
float64 matmul of the decoded operands, closed-form special cases (K = 1 outer
product, identity operand, all-maximum operands) and torch's CPU BF16 rounding
for the epilogue.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as o


def finite_codes(fmt, shape, rng, limit=None):
    table = o.fp8_decode_table(fmt)
    ok = np.nonzero(np.isfinite(table) & (np.abs(table) <= (limit or np.inf)))[0]
    return rng.choice(ok, size=shape).astype(np.uint8)


PAIRS = [(o.E4M3, o.E4M3), (o.E5M2, o.E4M3), (o.E5M2, o.E5M2), (o.E4M3, o.E5M2)]


@pytest.mark.parametrize("fa,fb", PAIRS)
def test_exact_path_against_fractions(fa, fb):
    rng = np.random.default_rng(10)
    A = finite_codes(fa, (3, 5), rng)
    B = finite_codes(fb, (4, 5), rng)
    ta, tb = o.fp8_decode_table(fa), o.fp8_decode_table(fb)
    acc = o.gemm_tn_exact(A, fa, B, fb)
    for i in range(3):
        for j in range(4):
            exact = sum(Fraction(ta[A[i, k]]) * Fraction(tb[B[j, k]]) for k in range(5))
            assert Fraction(acc[i, j]) == exact or \
                abs(Fraction(acc[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 53)


@pytest.mark.parametrize("fa,fb", PAIRS)
def test_double_path_against_numpy_and_exact(fa, fb):
    rng = np.random.default_rng(11)
    M, N, K = 33, 47, 96
    A = finite_codes(fa, (M, K), rng, limit=1e4)
    B = finite_codes(fb, (N, K), rng, limit=1e4)
    ta, tb = o.fp8_decode_table(fa), o.fp8_decode_table(fb)
    acc = o.gemm_tn(A, fa, B, fb)
    ref = ta[A] @ tb[B].T                              # numpy float64 matmul
    mag = np.abs(ta[A]) @ np.abs(tb[B]).T
    assert np.all(np.abs(acc - ref) <= mag * K * 2.0 ** -52)
    ex = o.gemm_tn_exact(A, fa, B, fb)
    assert np.all(np.abs(acc - ex) <= mag * K * 2.0 ** -52)
    # a block of rows equals the same rows of the full product
    part = o.gemm_tn(A, fa, B, fb, row0=10, nrows=7)
    assert np.array_equal(part, acc[10:17])


def test_special_cases():
    rng = np.random.default_rng(12)
    # K = 1 is an outer product
    A = finite_codes(o.E4M3, (6, 1), rng)
    B = finite_codes(o.E5M2, (9, 1), rng)
    ta, tb = o.fp8_decode_table(o.E4M3), o.fp8_decode_table(o.E5M2)
    assert np.array_equal(o.gemm_tn_exact(A, o.E4M3, B, o.E5M2), np.outer(ta[A[:, 0]], tb[B[:, 0]]))
    # identity operand (code 0x38 is 1.0 in E4M3) gives back the decoded A
    K = 16
    A = finite_codes(o.E4M3, (5, K), rng)
    I8 = np.where(np.eye(K, dtype=bool), 0x38, 0x00).astype(np.uint8)
    assert o.fp8_decode(0x38, o.E4M3) == 1.0
    assert np.array_equal(o.gemm_tn(A, o.E4M3, I8, o.E4M3), ta[A])
    # all-maximum operands: 448 * 448 * K and 57344 * 448 * K, exactly
    for fa, top in [(o.E4M3, 0x7E), (o.E5M2, 0x7B)]:
        A = np.full((2, 8192), top, np.uint8)
        B = np.full((3, 8192), 0xFE, np.uint8)   # -448
        acc = o.gemm_tn_exact(A, fa, B, o.E4M3)
        assert np.all(acc == -o.fp8_max(fa) * 448.0 * 8192)
        assert np.array_equal(o.gemm_tn(A, fa, B, o.E4M3), acc)


def test_epilogue_matches_torch_bf16_rounding():
    rng = np.random.default_rng(13)
    acc = rng.standard_normal(50000) * 10.0 ** rng.integers(-6, 6, 50000)
    sa, sb = np.float32(0.0123), np.float32(3.7e-3)
    y = o.epilogue(acc, sa, sb)
    sab = np.float32(sa * sb)
    v = (acc.astype(np.float32) * sab).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, ref)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _f(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_layer_step_approximates_the_real_linear():
    """Forward and backward of the FP8 layer stay within the FP8 rounding
    bound of the exact BF16 products: Y ~ X W^T, dX ~ dY W, dW ~ dY^T X.  A
    transposed operand or a wrong scale fails by orders of magnitude."""
    rng = np.random.default_rng(14)
    M, N, K = 32, 48, 64
    X = _bf16(rng.standard_normal((M, K)))
    W = _bf16(rng.standard_normal((N, K)) / 8)
    dY = _bf16(rng.standard_normal((M, N)) * 1e-3)
    rc = o.Recipe(margin=0, history_len=4)
    st = o.State.initial(4)
    # one step to learn the scales, then check the second (delayed) step
    for step in range(2):
        f = o.layer_fwd(st, rc, X, W)
        b = o.layer_bwd(st, rc, dY, f["X8t"], f["W8t"])
        if step == 1:
            Xd, Wd, dYd = _f(X), _f(W), _f(dY)
            for got, ref, mag, u in [
                (f["Y"], Xd @ Wd.T, np.abs(Xd) @ np.abs(Wd).T, 2 * 2.0 ** -4),
                (b["dX"], dYd @ Wd, np.abs(dYd) @ np.abs(Wd), 2.0 ** -3 + 2.0 ** -4),
                (b["dW"], dYd.T @ Xd, np.abs(dYd).T @ np.abs(Xd), 2.0 ** -3 + 2.0 ** -4),
            ]:
                err = np.abs(_f(got) - ref)
                assert np.all(err <= mag * (u + 2.0 ** -7) + 1e-30)
                assert np.linalg.norm(_f(got) - ref) / np.linalg.norm(ref) < 0.1
        o.layer_update(st, rc)
    assert st.history[o.SLOT_X, 0] == o.amax(X) and st.history[o.SLOT_X, 1] == o.amax(X)
    assert st.scale[o.SLOT_X] == np.float32(448.0) / o.amax(X)
    assert st.scale[o.SLOT_DY] == np.float32(57344.0) / o.amax(dY)
    assert st.amax[o.SLOT_Y] == o.amax(f["Y"])
