"""Shared helpers of the GPU parity tests: host copies, FP8 comparison with
NaN codes compared as a class, and the GEMM tolerance.

GEMM tolerance (per output tensor, against the oracle's BF16 output computed
with the same dequant epilogue): relative Frobenius error <= 1e-3 and
max |D_gpu - D_oracle| <= 2e-2 * sqrt(K) / 64 * max |D_oracle|.
"""
import math

import numpy as np
import torch

import oracle as o

FRO_TOL = 1e-3


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def f32_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def is_nan_code(q: np.ndarray, fmt: int) -> np.ndarray:
    m = q & 0x7F
    return (m == 0x7F) if fmt == o.E4M3 else (m > 0x7C)


def assert_fp8_equal(gpu: np.ndarray, ref: np.ndarray, fmt: int, what=""):
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    same = (gpu == ref) | (is_nan_code(gpu, fmt) & is_nan_code(ref, fmt))
    if not same.all():
        idx = np.argwhere(~same)[:5]
        raise AssertionError(f"{what}: {int((~same).sum())} FP8 codes differ, e.g. at "
                             f"{idx.tolist()}: gpu {[int(gpu[tuple(i)]) for i in idx]} "
                             f"oracle {[int(ref[tuple(i)]) for i in idx]}")


def gemm_errors(gpu_bits: np.ndarray, ref_bits: np.ndarray, K: int) -> dict:
    g, r = bf16_values(gpu_bits), bf16_values(ref_bits)
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    if nan_g.any() or nan_r.any():
        # NaN where, and only where, a NaN operand reaches the output
        if not np.array_equal(nan_g, nan_r):
            return dict(fro=np.inf, max_err=np.inf, bound=0.0, flips=-1, n=int(g.size),
                        nan_mismatch=int((nan_g != nan_r).sum()))
        g, r = g[~nan_r], r[~nan_r]
        gpu_bits, ref_bits = gpu_bits[~nan_r], ref_bits[~nan_r]
    diff = np.abs(g - r)
    ref_norm = np.linalg.norm(r)
    fro = float(np.linalg.norm(g - r) / ref_norm) if ref_norm > 0 else float(np.linalg.norm(g))
    scale = float(np.max(np.abs(r))) if r.size else 0.0
    bound = 2e-2 * math.sqrt(K) / 64 * scale
    return dict(fro=fro, max_err=float(diff.max()) if diff.size else 0.0, bound=bound,
                flips=int(np.count_nonzero(gpu_bits != ref_bits)), n=int(g.size))


def assert_gemm_close(gpu_bits, ref_bits, K, what=""):
    e = gemm_errors(gpu_bits, ref_bits, K)
    assert e["fro"] <= FRO_TOL and e["max_err"] <= e["bound"], (what, e)
    return e


def fp8_code_band(v: np.ndarray, tol: np.ndarray, fmt: int):
    """For a value v computed exactly (double) and an absolute error band tol
    of the float computation that produces it on the GPU, the FP8 codes a
    correct cast of any value in [v - tol, v + tol] can give: (expected code of
    v, code of v - tol, code of v + tol).  The cast is monotone, so a code is
    acceptable when its value lies between those of the two ends."""
    v = np.asarray(v, np.float64)
    tol = np.broadcast_to(np.asarray(tol, np.float64), v.shape)
    exp = o.fp8_encode(v.astype(np.float32), fmt).reshape(v.shape)
    lo = o.fp8_encode((v - tol).astype(np.float32), fmt).reshape(v.shape)
    hi = o.fp8_encode((v + tol).astype(np.float32), fmt).reshape(v.shape)
    return exp, lo, hi


def assert_codes_in_band(gpu: np.ndarray, v: np.ndarray, tol, fmt: int, what="", rare=1e-4):
    table = o.fp8_decode_table(fmt)
    exp, lo, hi = fp8_code_band(v, tol, fmt)
    g = table[gpu]
    ok = (gpu == exp) | ((g >= table[lo]) & (g <= table[hi]))
    assert ok.all(), (what, int((~ok).sum()), np.argwhere(~ok)[:5].tolist())
    differ = int((gpu != exp).sum())
    assert differ <= max(2, int(rare * gpu.size)), (what, differ)
    return differ


# ------------------------------------------------ full-size cast checks --

_CODE_TABLES = {}


def oracle_code_table(scale, fmt: int) -> np.ndarray:
    """The oracle's FP8 code of every BF16 bit pattern under ``scale``: its
    scaled cast (o.quantize) applied to all 65,536 patterns.  The cast is
    elementwise, so table[x_bits] is the oracle's cast of a whole tensor and
    table[x_bits].T its transposed copy.  Cached per (scale bits, format)."""
    key = (int(np.float32(scale).view(np.uint32)), int(fmt))
    t = _CODE_TABLES.get(key)
    if t is None:
        bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(1, -1)
        q, _ = o.quantize(bits, np.float32(scale), fmt, transpose=False)
        t = q.reshape(-1)
        t.setflags(write=False)
        if len(_CODE_TABLES) > 4096:
            _CODE_TABLES.clear()
        _CODE_TABLES[key] = t
    return t


def oracle_codes_host(x_bits: np.ndarray, table: np.ndarray) -> np.ndarray:
    """The oracle's codes of a host BF16 tensor through its code table."""
    return table[x_bits]


def assert_codes_on_device(gpu_codes, x, table: np.ndarray, fmt: int, transposed=False, what=""):
    """Every FP8 byte of a GPU cast output against the oracle's codes of the
    same BF16 input (through its 65,536-entry table; the lookup and the
    comparison run on the device, the values are the oracle's), NaN codes
    compared as a class.  ``transposed``: gpu_codes is the [cols, rows] copy."""
    import torch
    t = torch.from_numpy(np.array(table, copy=True)).to(gpu_codes.device)
    idx = x.contiguous().view(torch.int16).to(torch.int64) & 0xFFFF
    exp = t[idx]
    if transposed:
        exp = exp.t()
    g = gpu_codes.view(torch.uint8)
    assert tuple(g.shape) == tuple(exp.shape), (what, tuple(g.shape), tuple(exp.shape))
    diff = g != exp
    if bool(diff.any()):
        def nan_code(c):
            m = c & 0x7F
            return (m == 0x7F) if fmt == o.E4M3 else (m > 0x7C)
        bad = diff & ~(nan_code(g) & nan_code(exp))
        nbad = int(bad.sum())
        if nbad:
            where = torch.nonzero(bad)[:5].cpu().tolist()
            raise AssertionError(f"{what}: {nbad} FP8 codes differ from the oracle's, e.g. at "
                                 f"{where}")


def device_absmax_bits(t) -> np.float32:
    """max |t| over a BF16 tensor with NaN skipped (0 when all NaN), as the
    exact float32 -- a property of the GPU's own output."""
    import torch
    a = t.float().abs()
    a = torch.where(torch.isnan(a), torch.zeros_like(a), a)
    return np.float32(a.max().item()) if a.numel() else np.float32(0.0)
