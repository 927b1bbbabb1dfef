"""GPU parity of the FP8 all-reduce with one shared scale (wiki note, bullet
"per-tensor scaling is the key": s'_g = min(s'_1 .. s'_N)).

* fp8_dequant_sum against the oracle (the exact sum times 1 / scale, rounded
  once to BF16), bit-exact, for 1..8 parts, special codes, extreme and
  non-finite scales, and a case where rounding twice would differ;
* the whole product path (fp8_allreduce: amax, own scale, MIN all-reduce,
  cast, all-to-all of FP8 code shards, decode-and-sum of this rank's shard,
  all-gather of the BF16 shards) as 2 and 3 gloo ranks that share cuda:0 --
  their kernels never wait on one another, the exchange runs on the host --
  against the oracle's all-reduce, bit-exact on every rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as o

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
@pytest.mark.parametrize("nranks", [1, 2, 5, 8])
def test_dequant_sum_bit_exact(fmt, nranks):
    import fp8_mixed_precision_amax_gb300 as f
    rng = np.random.default_rng(10 * nranks + fmt)
    table = o.fp8_decode_table(fmt)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    n = 65536 + 16
    parts = rng.choice(finite, size=(nranks, n))
    s = np.float32(10.0 ** rng.uniform(-3, 3))
    out = torch.full((n,), float("nan"), dtype=torch.bfloat16, device="cuda")
    f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), fmt, torch.tensor([s], device="cuda"), out)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(out), o.dequant_sum(parts, fmt, s))


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
@pytest.mark.parametrize("nranks", [9, 64, 300, 1000])
def test_dequant_sum_many_ranks(fmt, nranks):
    """More than 8 ranks: the sums become int64 counts of quanta after every
    stage of 8 ranks; beyond 256 ranks the general path multiplies with 128
    bits.  Random finite codes, then every rank at the largest magnitude of
    one sign (1000 x 57344 x 2^16 quanta needs more than 40 bits), at
    ordinary, overflowing and BF16-subnormal scales; bit-exact."""
    import fp8_mixed_precision_amax_gb300 as f
    rng = np.random.default_rng(nranks + 17 * fmt)
    table = o.fp8_decode_table(fmt)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    top = 0x7E if fmt == o.E4M3 else 0x7B
    n = 4096 + 16
    cases = [rng.choice(finite, size=(nranks, n)),
             np.where(np.arange(n)[None, :] % 2 == 0, top, top | 0x80).repeat(nranks, 0)
             .astype(np.uint8)]
    for parts in cases:
        dev = torch.from_numpy(np.ascontiguousarray(parts)).cuda()
        for s in (np.float32(10.0 ** rng.uniform(-2, 2)), np.float32(1e-36), np.float32(1e36),
                  np.float32(-0.7)):
            out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
            f.fp8_dequant_sum(dev, fmt, torch.tensor([s], device="cuda"), out)
            torch.cuda.synchronize()
            assert _same_bf16(_u16(out), o.dequant_sum(parts, fmt, s)), (nranks, s)


def test_dequant_sum_rounds_once():
    """E5M2 parts 57344 + 128 + 2^-16 at scale 1: the exact sum lies just
    above the midpoint between the BF16 neighbours 57344 and 57600, so one
    rounding gives 57600 (0x4761); the parts without 2^-16 are the midpoint
    itself, which ties to the even 57344 (0x4760)."""
    import fp8_mixed_precision_amax_gb300 as f
    parts = np.zeros((3, 16), np.uint8)
    parts[:, 0] = [0x7B, 0x58, 0x01]
    parts[:2, 1] = [0x7B, 0x58]
    out = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), o.E5M2, torch.ones(1, device="cuda"), out)
    torch.cuda.synchronize()
    got = _u16(out)
    assert got[0] == 0x4761 and got[1] == 0x4760
    assert np.array_equal(got, o.dequant_sum(parts, o.E5M2, np.float32(1.0)))


def _same_bf16(a, b):
    """Equal BF16 bits, NaN compared as a class."""
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b])


@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_dequant_sum_specials_and_extremes(fmt):
    """Infinities and NaN among the parts follow IEEE arithmetic (NaN, or
    +inf with -inf, give NaN); 64 ranks of the largest magnitudes and mixed
    signs stay exact; a 4 M-element case runs several grid-stride passes of
    the kernel; scales whose results overflow BF16, land in its subnormal
    range or underflow, and zero, infinite, negative and NaN scales."""
    import fp8_mixed_precision_amax_gb300 as f
    rng = np.random.default_rng(7 + fmt)
    table = o.fp8_decode_table(fmt)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    specials = np.nonzero(~np.isfinite(table))[0].astype(np.uint8)
    top = 0x7E if fmt == o.E4M3 else 0x7B
    cases = []
    # sprinkle every special code into random finite parts
    parts = rng.choice(finite, size=(5, 4096))
    for j, c in enumerate(specials):
        parts[j % 5, rng.integers(0, 4096, 64)] = c
    cases.append(parts)
    if fmt == o.E5M2:   # +inf and -inf in the same element, and each alone
        p2 = rng.choice(finite, size=(3, 64))
        p2[0, :16], p2[1, :16] = 0x7C, 0xFC
        p2[0, 16:32] = 0x7C
        p2[2, 32:48] = 0xFC
        cases.append(p2)
    cases.append(np.where(rng.random((64, 2048)) < 0.5, top, top | 0x80).astype(np.uint8))
    cases.append(np.full((64, 1024), top, np.uint8))
    cases.append(rng.choice(finite, size=(3, (1 << 22) + 16)))
    scales = [np.float32(1e-30), np.float32(3e38), np.float32(1e36), np.float32(2.0 ** -100),
              np.float32(2.0 ** -125 * 1.3), np.float32(1e-45), np.float32(0.0),
              np.float32(np.inf), np.float32(-3.0), np.float32(np.nan), np.float32(2.0 ** 120)]
    for ci, parts in enumerate(cases):
        s = np.float32(10.0 ** rng.uniform(-4, 2))
        out = torch.empty(parts.shape[1], dtype=torch.bfloat16, device="cuda")
        f.fp8_dequant_sum(torch.from_numpy(np.ascontiguousarray(parts)).cuda(), fmt,
                          torch.tensor([s], device="cuda"), out)
        torch.cuda.synchronize()
        assert _same_bf16(_u16(out), o.dequant_sum(parts, fmt, s)), parts.shape
    # results past FLT_MAX, in the fp32 subnormal range and at its edge
    parts = rng.choice(finite, size=(4, 8192))
    for s in scales:
        out = torch.empty(parts.shape[1], dtype=torch.bfloat16, device="cuda")
        f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), fmt, torch.tensor([s], device="cuda"),
                          out)
        torch.cuda.synchronize()
        assert _same_bf16(_u16(out), o.dequant_sum(parts, fmt, s)), s


def _grads(world, shape, seed):
    out = []
    for r in range(world):
        g = torch.Generator().manual_seed(seed + r)
        out.append((torch.randn(shape, generator=g) * 10.0 ** (-3 + r)).to(torch.bfloat16))
    return out


@pytest.mark.parametrize("nranks", [1, 3, 8])
def test_dequant_sum_unsplit_e5m2_sums(nranks):
    """E5M2 values that are zero or at least 2^-3 in magnitude are multiples
    of 2^-5, so up to 8 of them add exactly in one fp32 sum; a nonzero value
    below 2^-3 is not.  Threads whose 16 elements hold only the former take
    the unsplit sum: here most do, a few elements carry one small code (so a
    warp mixes both kinds), some cancel to an exact zero, some hold infinities
    or NaN; the scales reach overflow, BF16's subnormal range, zero, negative
    and non-finite factors.  Gradient-shaped codes (N(0, sigma_r) cast at a
    shared scale, as the all-reduce makes them) follow."""
    import fp8_mixed_precision_amax_gb300 as f
    rng = np.random.default_rng(40 + nranks)
    table = o.fp8_decode_table(o.E5M2)
    finite = np.isfinite(table)
    small = finite & (table != 0) & (np.abs(table) < 0.125)
    big = np.nonzero(finite & ~small)[0].astype(np.uint8)
    tiny = np.nonzero(small)[0].astype(np.uint8)
    n = 8 * 4096 + 16
    parts = rng.choice(big, size=(nranks, n))
    k = np.arange(n)
    sel = (k % 997 == 5)
    parts[rng.integers(0, nranks, sel.sum()), k[sel]] = rng.choice(tiny, sel.sum())
    if nranks >= 2:
        z = (k % 61 == 7)
        parts[:, z] = 0
        parts[0, z] = rng.choice(big, z.sum())
        parts[1, z] = parts[0, z] ^ 0x80
    sp = (k % 1409 == 11)
    parts[rng.integers(0, nranks, sp.sum()), k[sp]] = rng.choice(
        np.array([0x7C, 0xFC, 0x7D, 0xFF], np.uint8), sp.sum())
    assert not np.isin(parts[:, k % 997 != 5], tiny).any()
    dev = torch.from_numpy(parts).cuda()
    scales = [np.float32(10.0 ** rng.uniform(-3, 3)), np.float32(1.0), np.float32(-3.0),
              np.float32(1e-30), np.float32(3e38), np.float32(2.0 ** -100),
              np.float32(2.0 ** 120), np.float32(1e-45), np.float32(0.0),
              np.float32(np.inf), np.float32(np.nan)]
    for s in scales:
        out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        f.fp8_dequant_sum(dev, o.E5M2, torch.tensor([s], device="cuda"), out)
        torch.cuda.synchronize()
        assert _same_bf16(_u16(out), o.dequant_sum(parts, o.E5M2, s)), s
    # gradient-shaped codes
    n = 1 << 18
    g = [rng.normal(0.0, 1e-3 * (1 + r / 10), n).astype(np.float32) for r in range(nranks)]
    s = np.float32(57344.0 / max(float(np.abs(x).max()) for x in g))
    parts = np.stack([o.quantize_f32(x, s, o.E5M2).reshape(-1) for x in g])
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), o.E5M2, torch.tensor([s], device="cuda"),
                      out)
    torch.cuda.synchronize()
    assert np.array_equal(_u16(out), o.dequant_sum(parts, o.E5M2, s))


@pytest.mark.parametrize("amax", [0.0057678, 1.0, 3.140625, 0.000244140625, 448.0])
def test_dequant_sum_recipe_scales(amax):
    """Scales as the recipe makes them, fl32(57344 / amax) for a BF16 amax:
    their inverses repeat the bits of 1/7, so the products of short exact
    sums land on and next to BF16 midpoints far more often than chance.
    Uniformly random codes (split sums that mostly do not add exactly in
    binary32, rounded through the rounding test) and gradient-shaped codes
    (exact unsplit sums) must both match the oracle bit for bit."""
    import fp8_mixed_precision_amax_gb300 as f
    rng = np.random.default_rng(int(amax * 1e6) % 1000 + 3)
    a16 = np.float32(torch.tensor(amax, dtype=torch.bfloat16).float().item())
    s = np.float32(np.float32(57344.0) / a16)
    n = 1 << 17
    table = o.fp8_decode_table(o.E5M2)
    finite = np.nonzero(np.isfinite(table))[0].astype(np.uint8)
    cases = [rng.choice(finite, size=(8, n))]
    g = [rng.normal(0.0, a16 / 5.5, n).astype(np.float32) for _ in range(8)]
    cases.append(np.stack([o.quantize_f32(x, s, o.E5M2).reshape(-1) for x in g]))
    for parts in cases:
        out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), o.E5M2, torch.tensor([s], device="cuda"),
                          out)
        torch.cuda.synchronize()
        assert _same_bf16(_u16(out), o.dequant_sum(parts, o.E5M2, s))


def test_dequant_sum_full_size_8_ranks_7b_dw():
    """The bench's FP8 all-reduce sum at full size: 8 ranks' N(0, sigma_r)
    gradients of the 7B layer's dW ([11008, 4096], sigma_r = 1e-3 (1 + r/10),
    BF16) cast to E5M2 with their shared scale (the minimum of the ranks'
    recipe scales), summed in one launch; every one of the 45 M outputs
    against the oracle, bit for bit."""
    import fp8_mixed_precision_amax_gb300 as f
    n = 11008 * 4096
    g = torch.Generator().manual_seed(8)
    grads = [(torch.randn(n, generator=g) * (1e-3 * (1 + 0.1 * r))).to(torch.bfloat16)
             for r in range(8)]
    scales = [np.float32(np.float32(57344.0) / np.float32(x.float().abs().max().item()))
              for x in grads]
    s = min(scales)
    parts = np.stack([o.quantize_f32(x.float().numpy(), s, o.E5M2).reshape(-1) for x in grads])
    del grads
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    f.fp8_dequant_sum(torch.from_numpy(parts).cuda(), o.E5M2, torch.tensor([s], device="cuda"),
                      out)
    f.fp8_sync_status()
    assert np.array_equal(_u16(out), o.dequant_sum(parts, o.E5M2, s))


def _worker(rank, world, port, shape, fmt, margin, q):
    import datetime

    import torch.distributed as dist
    import fp8_mixed_precision_amax_gb300 as f
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=60))
    try:
        grads = _grads(world, shape, 1234)
        out = f.fp8_allreduce(grads[rank].cuda(), fmt, margin)
        torch.cuda.synchronize()
        q.put((rank, _u16(out)))
    except Exception as e:   # reported to the parent
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("world,fmt,margin", [(2, o.E5M2, 0), (3, o.E4M3, 1)])
def test_allreduce_ranks_sharing_one_gpu(world, fmt, margin):
    shape = (272, 1040)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, shape, fmt, margin, q))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    grads = [_u16(g) for g in _grads(world, shape, 1234)]
    ref, sg, _ = o.fp8_allreduce(grads, fmt, margin)
    for r in range(world):
        assert not isinstance(res[r], str), res[r]
        assert np.array_equal(res[r].reshape(-1), ref), r
