"""GPU parity of the tcgen05 FP8 GEMM + dequant epilogue against the oracle.

Outputs are compared with the oracle's BF16 output (same epilogue) within
the tolerance in helpers.py; the fused output amax must equal max |D| over
the GPU's own BF16 output exactly, and match the oracle's within one BF16
rounding.  Shapes cover a single tile, several tiles, ragged M / N / K tails
and long K, for every operand-format pair.
"""
import numpy as np
import pytest
import torch

import oracle as o
from helpers import assert_gemm_close, bf16_values, f32_bits, host_bf16_bits

pytestmark = pytest.mark.gpu

PAIRS = [(o.E4M3, o.E4M3), (o.E5M2, o.E4M3), (o.E4M3, o.E5M2), (o.E5M2, o.E5M2)]


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _codes(shape, fmt, std, seed):
    """FP8 operands made the way the layer makes them: a scaled cast of
    Gaussian data (so magnitudes follow a realistic spread)."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * std).to(torch.bfloat16)
    q, _ = o.quantize(host_bf16_bits(x), np.float32(1.0), fmt, transpose=False)
    return q


def _run(A, fa, B, fb, sa, sb):
    f = _lib()
    M, K = A.shape
    N = B.shape[0]
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    am = torch.full((1,), -1.0, device="cuda")
    f.fp8_gemm_tn(dA, fa, dB, fb, torch.tensor([sa], device="cuda"),
                  torch.tensor([sb], device="cuda"), D, am)
    f.fp8_sync_status()
    return host_bf16_bits(D), np.float32(am.cpu().numpy()[0])


SHAPES = [(16, 16, 16), (128, 256, 128), (256, 256, 256), (144, 272, 48), (384, 512, 1040),
          (1040, 784, 400), (128, 256, 4096)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("fa,fb", PAIRS)
def test_gemm_matches_oracle(M, N, K, fa, fb):
    A = _codes((M, K), fa, 3.0 if fa == o.E4M3 else 300.0, M * 3 + K)
    B = _codes((N, K), fb, 1.0, N * 5 + K)
    sa, sb = np.float32(0.013), np.float32(0.77)
    got, am = _run(A, fa, B, fb, sa, sb)
    acc = o.gemm_tn(A, fa, B, fb)
    ref = o.epilogue(acc, sa, sb)
    e = assert_gemm_close(got, ref, K, f"{M}x{N}x{K} {fa}{fb}")
    # fused amax == max |D| of the emitted output, exactly; and near the oracle's
    assert f32_bits(am) == f32_bits(np.float32(np.max(np.abs(bf16_values(got))))), e
    assert abs(float(am) - float(np.max(np.abs(bf16_values(ref))))) <= e["bound"] + 1e-30


def test_gemm_exact_small_integers():
    """Operands whose products and sums are exact in fp32 (small integers):
    the GPU must reproduce the exact result bit for bit."""
    rng = np.random.default_rng(3)
    M, N, K = 256, 512, 384
    vals = np.array([0, 1, 2, 3, 4, -1, -2, -3, -4], np.float32)
    A = o.fp8_encode(rng.choice(vals, (M, K)), o.E4M3).reshape(M, K)
    B = o.fp8_encode(rng.choice(vals, (N, K)), o.E5M2).reshape(N, K)
    got, _ = _run(A, o.E4M3, B, o.E5M2, np.float32(1.0), np.float32(1.0))
    ref = o.epilogue(o.gemm_tn_exact(A, o.E4M3, B, o.E5M2), 1.0, 1.0)
    assert np.array_equal(got, ref)


def test_gemm_extreme_operands_and_zero():
    M, N, K = 128, 256, 256
    A = np.full((M, K), 0x7E, np.uint8)                  # +448
    B = np.full((N, K), 0xFB, np.uint8)                  # -57344 in E5M2
    got, am = _run(A, o.E4M3, B, o.E5M2, np.float32(2.0 ** -20), np.float32(1.0))
    ref = o.epilogue(o.gemm_tn_exact(A, o.E4M3, B, o.E5M2), 2.0 ** -20, 1.0)
    assert np.array_equal(got, ref)
    Z = np.zeros((M, K), np.uint8)
    got, am = _run(Z, o.E4M3, B, o.E5M2, np.float32(1.0), np.float32(1.0))
    assert np.all((got & 0x7FFF) == 0) and am == 0.0


def test_gemm_sync_status_clean():
    f = _lib()
    f.fp8_sync_status()


@pytest.mark.parametrize("shapes", [((384, 512, 1040), (1040, 784, 400)),
                                    ((128, 256, 128), (400, 272, 48)),
                                    ((8192, 4096, 512), (4096, 1024, 8192))])
def test_grouped_launch_matches_oracle(shapes):
    """Two independent GEMMs in one launch (as the backward pass runs dgrad and
    wgrad): each result matches its own oracle product, each amax its output."""
    f = _lib()
    probs, refs = [], []
    for i, ((M, N, K), (fa, fb)) in enumerate(zip(shapes, [(o.E5M2, o.E4M3), (o.E4M3, o.E5M2)])):
        A = _codes((M, K), fa, 300.0 if fa == o.E5M2 else 3.0, 11 * M + K + i)
        B = _codes((N, K), fb, 1.0, 13 * N + K + i)
        sa, sb = np.float32(0.011 * (i + 1)), np.float32(0.5)
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        am = torch.full((1,), -1.0, device="cuda")
        probs.append((torch.from_numpy(A).cuda(), fa, torch.from_numpy(B).cuda(), fb,
                      torch.tensor([sa], device="cuda"), torch.tensor([sb], device="cuda"), D, am))
        if M > 1024:   # sampled rows of the big ones
            rows = [(0, 16), (M // 2, 16), (M - 16, 16)]
            refs.append((K, [(r0, o.epilogue(o.gemm_tn(A, fa, B, fb, r0, n), sa, sb))
                             for r0, n in rows]))
        else:
            refs.append((K, [(0, o.epilogue(o.gemm_tn(A, fa, B, fb), sa, sb))]))
    f.fp8_gemm_tn_grouped(probs)
    f.fp8_sync_status()
    for (A, fa, B, fb, sa, sb, D, am), (K, blocks) in zip(probs, refs):
        got = host_bf16_bits(D)
        for r0, ref in blocks:
            assert_gemm_close(got[r0:r0 + ref.shape[0]], ref, K, f"{tuple(D.shape)} rows {r0}")
        full_max = np.float32(np.max(np.abs(bf16_values(got))))
        assert f32_bits(np.float32(am.item())) == f32_bits(full_max)


def test_gemm_degenerate_dequant_factors():
    """The ABI takes any scale_inv, so fl32(a_scale_inv * b_scale_inv) may be
    0, inf, NaN or underflow to 0.  With small-integer operands the fp32
    accumulation is exact, so every output is fixed by IEEE arithmetic: D
    matches the oracle's epilogue bit for bit (BF16 NaN as a class), and the
    fused amax is max |D| over the non-NaN outputs (infinities included; 0
    when every output is NaN)."""
    rng = np.random.default_rng(17)
    M, N, K = 128, 256, 64
    vals = np.array([0, 1, 2, 3, 4, -1, -2, -3, -4], np.float32)
    A = o.fp8_encode(rng.choice(vals, (M, K)), o.E4M3).reshape(M, K)
    B = o.fp8_encode(rng.choice(vals, (N, K)), o.E4M3).reshape(N, K)
    acc = o.gemm_tn_exact(A, o.E4M3, B, o.E4M3)
    assert (acc == 0).any() and (acc > 0).any() and (acc < 0).any()
    nan16 = lambda b: (b & 0x7FFF) > 0x7F80
    for sa, sb in ((0.0, 1.0), (float("inf"), 1.0), (float("nan"), 2.0), (1e30, 1e30),
                   (1e-30, 1e-30), (-float("inf"), 0.5)):
        got, am = _run(A, o.E4M3, B, o.E4M3, np.float32(sa), np.float32(sb))
        ref = o.epilogue(acc, np.float32(sa), np.float32(sb))
        both_nan = nan16(got) & nan16(ref)
        assert np.array_equal(nan16(got), nan16(ref)), (sa, sb)
        assert np.array_equal(got[~both_nan], ref[~both_nan]), (sa, sb)
        vals_ok = np.abs(bf16_values(got[~nan16(got)]))
        expect = np.float32(vals_ok.max()) if vals_ok.size else np.float32(0.0)
        assert f32_bits(am) == f32_bits(expect), (sa, sb, am, expect)


def test_clock_probe_measures_the_gemm_clock():
    """The diagnostic clock probe: while set, every GEMM launch adds its first
    CTA's SM cycles and nanoseconds; the ratio is a plausible SM clock (the
    part's maximum is 2.07 GHz); once cleared, launches add nothing."""
    import fp8_mixed_precision_amax_gb300 as f
    M, N, K = 1024, 2048, 4096
    g = torch.Generator().manual_seed(5)
    A = torch.randint(0, 0x7E, (M, K), generator=g, dtype=torch.uint8).cuda()
    B = torch.randint(0, 0x7E, (N, K), generator=g, dtype=torch.uint8).cuda()
    one = torch.ones(1, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    acc = torch.zeros(2, dtype=torch.int64, device="cuda")
    f.fp8_set_clock_probe(acc)
    try:
        for _ in range(5):
            f.fp8_gemm_tn(A, f.E4M3, B, f.E4M3, one, one, D)
    finally:
        f.fp8_set_clock_probe(None)
    torch.cuda.synchronize()
    cyc, ns = (int(v) for v in acc.cpu())
    assert cyc > 0 and ns > 0
    assert 0.3 < cyc / ns < 2.2, (cyc, ns)
    f.fp8_gemm_tn(A, f.E4M3, B, f.E4M3, one, one, D)
    torch.cuda.synchronize()
    assert [int(v) for v in acc.cpu()] == [cyc, ns]
    f.fp8_sync_status()
