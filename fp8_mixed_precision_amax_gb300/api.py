"""Python binding of the C ABI in include/fp8amax.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  It checks
that the torch tensors it is given are CUDA tensors of the right dtype,
shape and layout, passes their device pointers and the current torch CUDA
stream to the library, and raises ``Fp8Error`` on a non-OK status.  Every
step of the computation runs in the library's sm_103a kernels; there is no
fallback: if ``libfp8amax.so`` is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import logging
import os
import re
from dataclasses import dataclass

import torch

_log = logging.getLogger(__name__)
_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp8amax.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "fp8amax.h")

E4M3, E5M2 = 0, 1
SLOT_X, SLOT_W, SLOT_Y, SLOT_DY, SLOT_DX = range(5)
NUM_SLOTS = 5
STATUS = {0: "FP8_OK", 1: "FP8_ERR_ARG", 2: "FP8_ERR_ALIGN", 3: "FP8_ERR_CUDA",
          4: "FP8_ERR_TIMEOUT", 5: "FP8_ERR_UNSUPPORTED"}


class Fp8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class fp8_meta(ctypes.Structure):
    _fields_ = [("history", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("scale_inv", ctypes.c_void_p),
                ("history_len", ctypes.c_int32)]


class fp8_recipe(ctypes.Structure):
    _fields_ = [("margin", ctypes.c_int32), ("history_len", ctypes.c_int32),
                ("hybrid", ctypes.c_int32), ("scaling", ctypes.c_int32)]


SCALING_DELAYED, SCALING_CURRENT = 0, 1


class fp8_gemm_desc(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("fa", ctypes.c_int32), ("B", ctypes.c_void_p),
                ("fb", ctypes.c_int32), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("a_scale_inv", ctypes.c_void_p),
                ("b_scale_inv", ctypes.c_void_p), ("D", ctypes.c_void_p), ("d_amax", ctypes.c_void_p)]


class fp8_cast_desc(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("scale", ctypes.c_void_p), ("out", ctypes.c_void_p), ("out_t", ctypes.c_void_p),
                ("amax", ctypes.c_void_p)]


class fp8_adam_hyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("bias_correction1", ctypes.c_float), ("bias_correction2", ctypes.c_float),
                ("margin", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; call fp8_mixed_precision_amax_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32
    sig = {
        "fp8_abi_version": ([], i32),
        "fp8_last_error": ([], ctypes.c_char_p),
        "fp8_sync_status": ([vp], ctypes.c_int),
        "fp8_amax": ([vp, i64, vp, vp], ctypes.c_int),
        "fp8_set_clock_probe": ([vp], ctypes.c_int),
        "fp8_selftest_wait_timeout": ([i64, vp], ctypes.c_int),
        "fp8_quantize_transpose": ([vp, i64, i64, vp, i32, vp, vp, vp, vp], ctypes.c_int),
        "fp8_quantize_f32": ([vp, i64, vp, i32, vp, vp, vp], ctypes.c_int),
        "fp8_quantize_transpose_current": ([vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp],
                                           ctypes.c_int),
        "fp8_scale_update": ([vp, vp, vp, vp, i32, i32, u32, i32, vp], ctypes.c_int),
        "fp8_amax_scale_update": ([ctypes.POINTER(fp8_meta), ctypes.POINTER(fp8_recipe), vp],
                                  ctypes.c_int),
        "fp8_gemm_tn": ([vp, i32, vp, i32, i64, i64, i64, vp, vp, vp, vp, vp], ctypes.c_int),
        "fp8_gemm_tn_grouped": ([ctypes.POINTER(fp8_gemm_desc), i32, vp], ctypes.c_int),
        "fp8_quantize_transpose_grouped": ([ctypes.POINTER(fp8_cast_desc), i32, i32, vp],
                                           ctypes.c_int),
        "fp8_linear_fwd": ([vp, vp, i64, i64, i64, ctypes.POINTER(fp8_meta),
                            ctypes.POINTER(fp8_recipe), vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "fp8_linear_bwd": ([vp, i64, i64, i64, ctypes.POINTER(fp8_meta),
                            ctypes.POINTER(fp8_recipe), vp, vp, vp, vp, vp, vp, vp],
                           ctypes.c_int),
        "fp8_layernorm_quantize_transpose": ([vp, vp, vp, i64, i64, ctypes.c_float, vp, i32, vp,
                                              vp, vp, vp, vp, vp], ctypes.c_int),
        "fp8_layernorm_stats": ([vp, vp, vp, i64, i64, ctypes.c_float, vp, vp, vp, vp],
                                ctypes.c_int),
        "fp8_layernorm_linear_fwd": ([vp, vp, vp, ctypes.c_float, vp, i64, i64, i64,
                                      ctypes.POINTER(fp8_meta), ctypes.POINTER(fp8_recipe), vp, vp,
                                      vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "fp8_dequant_sum": ([vp, i32, i64, i32, vp, vp, vp], ctypes.c_int),
        "fp8_adam_step": ([vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                           ctypes.POINTER(fp8_adam_hyper), vp], ctypes.c_int),
        "fp8_adam_init": ([vp, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
        "fp8_linear_bwd_noalloc": ([vp, i64, i64, i64, ctypes.POINTER(fp8_meta),
                                    ctypes.POINTER(fp8_recipe), vp, vp, vp, vp, vp],
                                   ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes, f.restype = args, res
    if lib.fp8_abi_version() != 4:
        raise ImportError("libfp8amax.so ABI version mismatch")
    return lib


_lib = _load()


def header_functions() -> list[str]:
    """Names of the functions include/fp8amax.h declares."""
    src = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fp8_\w+)\s*\(", src, re.M)))


def library() -> ctypes.CDLL:
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise Fp8Error(status, _lib.fp8_last_error().decode())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


_U8 = torch.uint8


def _fp8_view_ok(t):
    return t.dtype in (torch.uint8, torch.float8_e4m3fn, torch.float8_e5m2)


def _p8(t, name):
    if t is None:
        return None
    if not _fp8_view_ok(t):
        raise ValueError(f"{name} must hold FP8 codes (uint8 / float8), got {t.dtype}")
    return _ptr(t, None, name)


# ------------------------------------------------------------ entry points --

def fp8_sync_status(stream=None) -> None:
    _check(_lib.fp8_sync_status(_stream(stream)))


def fp8_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Diagnostic: a kernel whose bounded wait runs out after ``limit_ns``;
    the next fp8_sync_status raises Fp8Error with FP8_ERR_TIMEOUT."""
    _check(_lib.fp8_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def fp8_set_clock_probe(acc: torch.Tensor | None) -> None:
    """Diagnostic: while ``acc`` (a zeroed CUDA int64 tensor of 2) is set, the
    first CTA of every GEMM launch adds its SM cycles to acc[0] and its
    nanoseconds to acc[1]; acc[0] / acc[1] is the average SM clock in GHz.
    None turns the probe off."""
    if acc is not None and (acc.dtype != torch.int64 or acc.numel() < 2):
        raise ValueError("acc must be an int64 tensor of at least 2 elements")
    _check(_lib.fp8_set_clock_probe(_ptr(acc, torch.int64, "acc")))


def fp8_amax(x: torch.Tensor, amax: torch.Tensor, stream=None) -> None:
    _check(_lib.fp8_amax(_ptr(x, torch.bfloat16, "x"), x.numel(), _ptr(amax, torch.float32, "amax"),
                         _stream(stream)))


def fp8_quantize_f32(x: torch.Tensor, scale: torch.Tensor, fmt: int, out: torch.Tensor,
                     amax=None, stream=None) -> None:
    """Scaled cast of a contiguous fp32 tensor to FP8 codes (uint8, same
    number of elements), optionally overwriting amax with max |x|."""
    if out.numel() != x.numel():
        raise ValueError("out must have as many elements as x")
    _check(_lib.fp8_quantize_f32(_ptr(x, torch.float32, "x"), x.numel(),
                                 _ptr(scale, torch.float32, "scale"), fmt, _p8(out, "out"),
                                 _ptr(amax, torch.float32, "amax"), _stream(stream)))


def fp8_quantize_transpose(x: torch.Tensor, scale: torch.Tensor, fmt: int, out=None, out_t=None,
                           amax=None, stream=None) -> None:
    rows, cols = x.shape
    if out is not None and tuple(out.shape) != (rows, cols):
        raise ValueError("out must be [rows, cols]")
    if out_t is not None and tuple(out_t.shape) != (cols, rows):
        raise ValueError("out_t must be [cols, rows]")
    _check(_lib.fp8_quantize_transpose(_ptr(x, torch.bfloat16, "x"), rows, cols,
                                       _ptr(scale, torch.float32, "scale"), fmt, _p8(out, "out"),
                                       _p8(out_t, "out_t"), _ptr(amax, torch.float32, "amax"),
                                       _stream(stream)))


def fp8_quantize_transpose_current(x: torch.Tensor, fmt: int, margin: int, amax: torch.Tensor,
                                   scale: torch.Tensor, scale_inv: torch.Tensor, out=None,
                                   out_t=None, stream=None) -> None:
    rows, cols = x.shape
    if out is not None and tuple(out.shape) != (rows, cols):
        raise ValueError("out must be [rows, cols]")
    if out_t is not None and tuple(out_t.shape) != (cols, rows):
        raise ValueError("out_t must be [cols, rows]")
    _check(_lib.fp8_quantize_transpose_current(
        _ptr(x, torch.bfloat16, "x"), rows, cols, fmt, margin, _p8(out, "out"), _p8(out_t, "out_t"),
        _ptr(amax, torch.float32, "amax"), _ptr(scale, torch.float32, "scale"),
        _ptr(scale_inv, torch.float32, "scale_inv"), _stream(stream)))


def fp8_scale_update(history: torch.Tensor, amax: torch.Tensor, scale: torch.Tensor,
                     scale_inv: torch.Tensor, format_mask: int, margin: int, stream=None) -> None:
    n, L = history.shape
    _check(_lib.fp8_scale_update(_ptr(history, torch.float32, "history"),
                                 _ptr(amax, torch.float32, "amax"),
                                 _ptr(scale, torch.float32, "scale"),
                                 _ptr(scale_inv, torch.float32, "scale_inv"), n, L, format_mask,
                                 margin, _stream(stream)))


def fp8_gemm_tn(A: torch.Tensor, fa: int, B: torch.Tensor, fb: int, a_scale_inv: torch.Tensor,
                b_scale_inv: torch.Tensor, D: torch.Tensor, d_amax=None, stream=None) -> None:
    M, K = A.shape
    N, K2 = B.shape
    if K != K2 or tuple(D.shape) != (M, N):
        raise ValueError("shapes: A [M,K], B [N,K], D [M,N]")
    _check(_lib.fp8_gemm_tn(_p8(A, "A"), fa, _p8(B, "B"), fb, M, N, K,
                            _ptr(a_scale_inv, torch.float32, "a_scale_inv"),
                            _ptr(b_scale_inv, torch.float32, "b_scale_inv"),
                            _ptr(D, torch.bfloat16, "D"), _ptr(d_amax, torch.float32, "d_amax"),
                            _stream(stream)))


def _val(p):
    return None if p is None else p.value


def fp8_gemm_tn_grouped(problems, stream=None) -> None:
    """One or two GEMMs in one launch; ``problems`` = list of tuples
    (A, fa, B, fb, a_scale_inv, b_scale_inv, D, d_amax-or-None)."""
    if not 1 <= len(problems) <= 2:
        raise ValueError("one or two problems")
    arr = (fp8_gemm_desc * len(problems))()
    for i, (A, fa, B, fb, sa, sb, D, am) in enumerate(problems):
        M, K = A.shape
        N, K2 = B.shape
        if K != K2 or tuple(D.shape) != (M, N):
            raise ValueError("shapes: A [M,K], B [N,K], D [M,N]")
        arr[i] = fp8_gemm_desc(_val(_p8(A, "A")), fa, _val(_p8(B, "B")), fb, M, N, K,
                               _val(_ptr(sa, torch.float32, "a_scale_inv")),
                               _val(_ptr(sb, torch.float32, "b_scale_inv")),
                               _val(_ptr(D, torch.bfloat16, "D")),
                               _val(_ptr(am, torch.float32, "d_amax")))
    _check(_lib.fp8_gemm_tn_grouped(arr, len(problems), _stream(stream)))


def fp8_quantize_transpose_grouped(tensors, fmt: int, stream=None) -> None:
    """One or two casts of one format in one launch; ``tensors`` = list of
    tuples (x, scale, out-or-None, out_t-or-None, amax-or-None)."""
    if not 1 <= len(tensors) <= 2:
        raise ValueError("one or two tensors")
    arr = (fp8_cast_desc * len(tensors))()
    for i, (x, scale, out, out_t, am) in enumerate(tensors):
        rows, cols = x.shape
        arr[i] = fp8_cast_desc(_val(_ptr(x, torch.bfloat16, "x")), rows, cols,
                               _val(_ptr(scale, torch.float32, "scale")), _val(_p8(out, "out")),
                               _val(_p8(out_t, "out_t")), _val(_ptr(am, torch.float32, "amax")))
    _check(_lib.fp8_quantize_transpose_grouped(arr, len(tensors), fmt, _stream(stream)))


# ------------------------------------------------------------------ layer --

@dataclass
class Recipe:
    """DelayedScaling: margin (default 0), amax_history_len (default 1024),
    HYBRID (E4M3 forward, E5M2 backward) or E4M3 everywhere; ``current``
    switches X, W and dY to just-in-time scaling from their own amax."""
    margin: int = 0
    history_len: int = 1024
    hybrid: bool = True
    current: bool = False

    def c(self) -> fp8_recipe:
        return fp8_recipe(self.margin, self.history_len, 1 if self.hybrid else 0,
                          SCALING_CURRENT if self.current else SCALING_DELAYED)

    def describe(self) -> str:
        """The precision mode in words, as a layer logs it when it is built."""
        return (f"E4M3 forward, {'E5M2' if self.hybrid else 'E4M3'} backward, "
                f"{'just-in-time' if self.current else 'delayed'} scaling, margin "
                f"{self.margin}, amax history {self.history_len}")


class Meta:
    """Per-layer scaling state on the device: history [5, L], amax [5],
    scale [5], scale_inv [5] (fp32), initialised to 0 / 0 / 1 / 1."""

    def __init__(self, history_len: int, device="cuda"):
        self.history = torch.zeros((NUM_SLOTS, history_len), dtype=torch.float32, device=device)
        self.amax = torch.zeros(NUM_SLOTS, dtype=torch.float32, device=device)
        self.scale = torch.ones(NUM_SLOTS, dtype=torch.float32, device=device)
        self.scale_inv = torch.ones(NUM_SLOTS, dtype=torch.float32, device=device)
        self.history_len = history_len

    def c(self) -> fp8_meta:
        return fp8_meta(self.history.data_ptr(), self.amax.data_ptr(), self.scale.data_ptr(),
                        self.scale_inv.data_ptr(), self.history_len)

    def state_dict(self) -> dict:
        return {"history": self.history.clone(), "amax": self.amax.clone(),
                "scale": self.scale.clone(), "scale_inv": self.scale_inv.clone()}

    def load_state_dict(self, d: dict) -> None:
        for k in ("history", "amax", "scale", "scale_inv"):
            getattr(self, k).copy_(d[k])


def fp8_amax_scale_update(meta: Meta, recipe: Recipe, stream=None) -> None:
    m, r = meta.c(), recipe.c()
    _check(_lib.fp8_amax_scale_update(ctypes.byref(m), ctypes.byref(r), _stream(stream)))


def fp8_linear_fwd(X, W, meta: Meta, recipe: Recipe, X8, X8t, W8, W8t, Y, stream=None) -> None:
    M, K = X.shape
    N, K2 = W.shape
    if K != K2 or tuple(Y.shape) != (M, N):
        raise ValueError("shapes: X [M,K], W [N,K], Y [M,N]")
    for t, shp, nm in [(X8, (M, K), "X8"), (X8t, (K, M), "X8t"), (W8, (N, K), "W8"),
                       (W8t, (K, N), "W8t")]:
        if tuple(t.shape) != shp:
            raise ValueError(f"{nm} must be {list(shp)}")
    m, r = meta.c(), recipe.c()
    _check(_lib.fp8_linear_fwd(_ptr(X, torch.bfloat16, "X"), _ptr(W, torch.bfloat16, "W"), M, N, K,
                               ctypes.byref(m), ctypes.byref(r), _p8(X8, "X8"), _p8(X8t, "X8t"),
                               _p8(W8, "W8"), _p8(W8t, "W8t"), _ptr(Y, torch.bfloat16, "Y"),
                               _stream(stream)))


def fp8_layernorm_quantize_transpose(x, gamma, beta, eps: float, scale, fmt: int, mean, rstd,
                                     out=None, out_t=None, amax=None, stream=None) -> None:
    rows, cols = x.shape
    _check(_lib.fp8_layernorm_quantize_transpose(
        _ptr(x, torch.bfloat16, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
        _ptr(beta, torch.bfloat16, "beta"), rows, cols, float(eps),
        _ptr(scale, torch.float32, "scale"), fmt, _p8(out, "out"), _p8(out_t, "out_t"),
        _ptr(amax, torch.float32, "amax"), _ptr(mean, torch.float32, "mean"),
        _ptr(rstd, torch.float32, "rstd"), _stream(stream)))


def fp8_layernorm_stats(x, gamma, beta, eps: float, mean, rstd, amax=None, stream=None) -> None:
    rows, cols = x.shape
    _check(_lib.fp8_layernorm_stats(
        _ptr(x, torch.bfloat16, "x"), _ptr(gamma, torch.bfloat16, "gamma"),
        _ptr(beta, torch.bfloat16, "beta"), rows, cols, float(eps),
        _ptr(mean, torch.float32, "mean"), _ptr(rstd, torch.float32, "rstd"),
        _ptr(amax, torch.float32, "amax"), _stream(stream)))


def fp8_layernorm_linear_fwd(X, gamma, beta, eps: float, W, meta: "Meta", recipe: "Recipe", X8, X8t,
                             W8, W8t, Y, mean, rstd, stream=None) -> None:
    M, K = X.shape
    N, K2 = W.shape
    if K != K2 or tuple(Y.shape) != (M, N):
        raise ValueError("shapes: X [M,K], W [N,K], Y [M,N]")
    m, r = meta.c(), recipe.c()
    _check(_lib.fp8_layernorm_linear_fwd(
        _ptr(X, torch.bfloat16, "X"), _ptr(gamma, torch.bfloat16, "gamma"),
        _ptr(beta, torch.bfloat16, "beta"), float(eps), _ptr(W, torch.bfloat16, "W"), M, N, K,
        ctypes.byref(m), ctypes.byref(r), _p8(X8, "X8"), _p8(X8t, "X8t"), _p8(W8, "W8"),
        _p8(W8t, "W8t"), _ptr(Y, torch.bfloat16, "Y"), _ptr(mean, torch.float32, "mean"),
        _ptr(rstd, torch.float32, "rstd"), _stream(stream)))


def fp8_linear_bwd(dY, meta: Meta, recipe: Recipe, X8t, W8t, dY8, dY8t, dX, dW,
                   stream=None) -> None:
    M, N = dY.shape
    K = X8t.shape[0]
    for t, shp, nm in [(X8t, (K, M), "X8t"), (W8t, (K, N), "W8t"), (dY8, (M, N), "dY8"),
                       (dY8t, (N, M), "dY8t")]:
        if tuple(t.shape) != shp:
            raise ValueError(f"{nm} must be {list(shp)}")
    if tuple(dX.shape) != (M, K) or tuple(dW.shape) != (N, K):
        raise ValueError("dX must be [M,K] and dW [N,K]")
    m, r = meta.c(), recipe.c()
    _check(_lib.fp8_linear_bwd(_ptr(dY, torch.bfloat16, "dY"), M, N, K, ctypes.byref(m),
                               ctypes.byref(r), _p8(X8t, "X8t"), _p8(W8t, "W8t"),
                               _p8(dY8, "dY8"), _p8(dY8t, "dY8t"), _ptr(dX, torch.bfloat16, "dX"),
                               _ptr(dW, torch.bfloat16, "dW"), _stream(stream)))


def fp8_linear_bwd_noalloc(dY, meta: Meta, recipe: Recipe, X8t, W8t, dX, dW,
                           stream=None) -> None:
    """fp8_linear_bwd without the dY8 / dY8t work buffers, for callers that
    cannot allocate device memory: the library keeps them in a fixed 64 MiB
    device array (M * N <= 2^25).  Calls that overlap on the GPU race on that
    array; the first call on a device should come before any stream capture."""
    M, N = dY.shape
    K = X8t.shape[0]
    for t, shp, nm in [(X8t, (K, M), "X8t"), (W8t, (K, N), "W8t")]:
        if tuple(t.shape) != shp:
            raise ValueError(f"{nm} must be {list(shp)}")
    if tuple(dX.shape) != (M, K) or tuple(dW.shape) != (N, K):
        raise ValueError("dX must be [M,K] and dW [N,K]")
    m, r = meta.c(), recipe.c()
    _check(_lib.fp8_linear_bwd_noalloc(_ptr(dY, torch.bfloat16, "dY"), M, N, K, ctypes.byref(m),
                                       ctypes.byref(r), _p8(X8t, "X8t"), _p8(W8t, "W8t"),
                                       _ptr(dX, torch.bfloat16, "dX"),
                                       _ptr(dW, torch.bfloat16, "dW"), _stream(stream)))


class Fp8Linear:
    """One FP8 linear layer Y = X W^T with delayed per-tensor scaling (the
    te.Linear + fp8_autocast + DelayedScaling pattern): owns the weight, the
    scaling state and the FP8 buffers kept between forward and backward.
    ``step`` = forward, backward, then the recipe's scale update, all enqueued
    on the current stream with no host synchronisation."""

    def __init__(self, W: torch.Tensor, M: int, recipe: Recipe | None = None):
        self.recipe = recipe or Recipe()
        self.W = W
        N, K = W.shape
        _log.info("FP8 linear [%d x %d], up to %d tokens: %s", N, K, M, self.recipe.describe())
        dev = W.device
        self.M, self.N, self.K = M, N, K
        self.meta = Meta(self.recipe.history_len, dev)
        e = lambda *s: torch.empty(s, dtype=torch.uint8, device=dev)
        self.X8, self.X8t, self.W8, self.W8t = e(M, K), e(K, M), e(N, K), e(K, N)
        self.dY8, self.dY8t = e(M, N), e(N, M)
        b = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)
        self.Y, self.dX, self.dW = b(M, N), b(M, K), b(N, K)

    def forward(self, X: torch.Tensor, stream=None, Y: torch.Tensor | None = None) -> torch.Tensor:
        """Y = X W^T; written into ``Y`` if given, else into the layer's own buffer."""
        Y = self.Y if Y is None else Y
        fp8_linear_fwd(X, self.W, self.meta, self.recipe, self.X8, self.X8t, self.W8, self.W8t,
                       Y, stream)
        return Y

    def backward(self, dY: torch.Tensor, stream=None, dX: torch.Tensor | None = None,
                 dW: torch.Tensor | None = None):
        """dX = dY W and dW = dY^T X, into the given buffers or the layer's own."""
        dX = self.dX if dX is None else dX
        dW = self.dW if dW is None else dW
        fp8_linear_bwd(dY, self.meta, self.recipe, self.X8t, self.W8t, self.dY8, self.dY8t,
                       dX, dW, stream)
        return dX, dW

    def update(self, stream=None) -> None:
        fp8_amax_scale_update(self.meta, self.recipe, stream)

    def capture_step(self, X: torch.Tensor, dY: torch.Tensor, outs=None) -> "torch.cuda.CUDAGraph":
        """Record one whole step on these input (and output) buffers as a CUDA
        graph; ``graph.replay()`` then re-runs forward, backward and the
        update with one launch.  Every scale lives on the device, so replays
        follow the recipe exactly as eager steps do.  The step is run once
        eagerly first (kernel attributes and tensor maps are set up outside
        the capture) -- that warm-up step advances the scaling state."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.step(X, dY, outs=outs)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(X, dY, outs=outs)
        return g

    def step(self, X: torch.Tensor, dY: torch.Tensor, stream=None, outs=None):
        """Forward, backward and the recipe's update; ``outs`` = (Y, dX, dW)
        buffers to write instead of the layer's own."""
        Y, dX, dW = outs if outs is not None else (None, None, None)
        Y = self.forward(X, stream, Y)
        dX, dW = self.backward(dY, stream, dX, dW)
        self.update(stream)
        return Y, dX, dW


def allreduce_amax(meta: Meta, group=None) -> None:
    """Data-parallel replicas each see their own shard of tokens; before the
    scale update they take the MAX of the five amaxes over all ranks so every
    replica derives the same scales (max is exact and order-free, so the
    result is bit-identical on every rank).  Uses torch.distributed."""
    import torch.distributed as dist
    dist.all_reduce(meta.amax, op=dist.ReduceOp.MAX, group=group)


class Fp8LayerNormLinear(Fp8Linear):
    """LayerNorm in front of an FP8 linear (te.LayerNormLinear): the forward
    normalises X with gamma / beta and casts the result straight to E4M3
    (fp8_layernorm_linear_fwd); the backward is the linear's, on that FP8
    LayerNorm output.  mean / rstd are kept for a LayerNorm backward."""

    def __init__(self, W: torch.Tensor, M: int, gamma: torch.Tensor, beta: torch.Tensor,
                 eps: float = 1e-5, recipe: Recipe | None = None):
        super().__init__(W, M, recipe)
        self.gamma, self.beta, self.eps = gamma, beta, eps
        self.mean = torch.empty(M, dtype=torch.float32, device=W.device)
        self.rstd = torch.empty(M, dtype=torch.float32, device=W.device)

    def forward(self, X: torch.Tensor, stream=None, Y: torch.Tensor | None = None) -> torch.Tensor:
        Y = self.Y if Y is None else Y
        fp8_layernorm_linear_fwd(X, self.gamma, self.beta, self.eps, self.W, self.meta,
                                 self.recipe, self.X8, self.X8t, self.W8, self.W8t, Y, self.mean,
                                 self.rstd, stream)
        return Y


@dataclass
class AdamHyper:
    """Adam / AdamW hyper-parameters; ``margin`` is the state scales' margin."""
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    margin: int = 0

    def c(self, t: int) -> fp8_adam_hyper:
        return fp8_adam_hyper(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay,
                              1.0 - self.beta1 ** t, 1.0 - self.beta2 ** t, self.margin)


class Fp8AdamState:
    """Decoupled-precision Adam state of one parameter tensor (wiki note,
    bullet "precision decoupling"): first moment E4M3 with a per-tensor scale,
    second moment FP16, master weights FP16 with a per-tensor scale -- 5 bytes
    of state per parameter.  ``scales`` = [m1_scale, m1_scale_inv, w_scale, w_scale_inv]."""

    def __init__(self, w: torch.Tensor, margin: int = 0, stream=None):
        """State of the BF16 weight tensor ``w``, initialised on the device by
        fp8_adam_init: zero moments, master weights FP16 under the
        just-in-time scale of w (fmax 65504, ``margin``)."""
        n = w.numel()
        dev = w.device
        self.n = n
        self.m1 = torch.empty(n, dtype=torch.uint8, device=dev)
        self.m2 = torch.empty(n, dtype=torch.float16, device=dev)
        self.w16 = torch.empty(n, dtype=torch.float16, device=dev)
        self.scales = torch.empty(4, dtype=torch.float32, device=dev)
        self.amax = torch.empty(2, dtype=torch.float32, device=dev)
        self.t = 0
        sc = self.scales
        wc = w.detach().reshape(-1)
        _check(_lib.fp8_adam_init(
            _ptr(wc, torch.bfloat16, "w"), n, int(margin), _p8(self.m1, "m1"),
            ctypes.c_void_p(sc.data_ptr()), ctypes.c_void_p(sc.data_ptr() + 4),
            _ptr(self.m2, torch.float16, "m2"), _ptr(self.w16, torch.float16, "w16"),
            ctypes.c_void_p(sc.data_ptr() + 8), ctypes.c_void_p(sc.data_ptr() + 12),
            _ptr(self.amax, torch.float32, "amax"), _stream(stream)))

    def step(self, grad: torch.Tensor, w_bf16: torch.Tensor, hp: AdamHyper, stream=None) -> None:
        """One step with ``grad`` (BF16, n elements); writes the new weights
        into ``w_bf16`` (BF16, n elements)."""
        if grad.numel() != self.n or w_bf16.numel() != self.n:
            raise ValueError("grad and w_bf16 must have the state's number of elements")
        self.t += 1
        h = hp.c(self.t)
        sc = self.scales
        _check(_lib.fp8_adam_step(
            _ptr(grad, torch.bfloat16, "grad"), self.n, _p8(self.m1, "m1"),
            ctypes.c_void_p(sc.data_ptr()), ctypes.c_void_p(sc.data_ptr() + 4),
            _ptr(self.m2, torch.float16, "m2"), _ptr(self.w16, torch.float16, "w16"),
            ctypes.c_void_p(sc.data_ptr() + 8), ctypes.c_void_p(sc.data_ptr() + 12),
            _ptr(w_bf16, torch.bfloat16, "w_bf16"), _ptr(self.amax, torch.float32, "amax"),
            ctypes.byref(h), _stream(stream)))


def fp8_dequant_sum(parts: torch.Tensor, fmt: int, scale: torch.Tensor, out: torch.Tensor,
                    stream=None) -> None:
    """out = BF16 of the sum over ranks of parts [nranks, n] (FP8 codes sharing
    one scale) times 1 / scale."""
    nranks, n = parts.shape
    if out.numel() != n:
        raise ValueError("out must hold n elements")
    _check(_lib.fp8_dequant_sum(_p8(parts, "parts"), nranks, n, fmt,
                                _ptr(scale, torch.float32, "scale"),
                                _ptr(out, torch.bfloat16, "out"), _stream(stream)))


def fp8_shard_len(n: int, world: int) -> int:
    """Elements per rank's shard in the FP8 all-reduce: n / world rounded up
    to a multiple of 16 (the library's alignment unit)."""
    per = -(-n // world)
    return -(-per // 16) * 16


def fp8_exchange_sum(q: torch.Tensor, shard: int, reduce_shard, group=None) -> torch.Tensor:
    """The exchange of the FP8 all-reduce as a reduce-scatter plus an
    all-gather, on codes every rank has cast with the one shared scale.

    ``q`` is this rank's [world * shard] FP8 codes (padded with code 0, +0).
    An all-to-all sends shard j to rank j, so every rank receives its own
    shard from all ranks, in rank order ([world, shard]); ``reduce_shard``
    turns those codes into the shard's reduced values ([shard], BF16); an
    all-gather of the reduced shards gives every rank the whole result
    ([world * shard]).  Each rank receives (world - 1) * shard FP8 bytes and
    (world - 1) * shard BF16 values: 3 (N - 1) / N bytes per element, against
    4 (N - 1) / N for a BF16 ring all-reduce and (N - 1) for an all-gather of
    every rank's codes.  Uses torch.distributed."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    if q.numel() != world * shard:
        raise ValueError("q must hold world * shard codes")
    recv = torch.empty_like(q)
    dist.all_to_all_single(recv, q, group=group)
    mine = reduce_shard(recv.view(world, shard))
    full = torch.empty(world * shard, dtype=mine.dtype, device=mine.device)
    dist.all_gather([full[r * shard:(r + 1) * shard] for r in range(world)], mine, group=group)
    return full


def fp8_allreduce(grad: torch.Tensor, fmt: int, margin: int = 0, group=None,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """All-reduce (sum) of a BF16 gradient [rows, cols] over the ranks of
    ``group`` with FP8 communication and one scale shared by all ranks, the
    minimum of the ranks' own scales (wiki note, bullet "per-tensor scaling is
    the key"):
      1. this rank's scale: amax, then the recipe formula on a one-entry history;
      2. the shared scale: all-reduce(MIN) of the scales;
      3. the cast of the gradient with the shared scale (fp8_quantize_transpose);
      4. reduce-scatter: all-to-all of the FP8 codes by shard, then
         fp8_dequant_sum of this rank's shard (the exact sum of all ranks'
         values times 1 / scale, rounded once to BF16);
      5. all-gather of the reduced BF16 shards.
    Every rank ends with the same result, the oracle's sum bit for bit.
    Uses torch.distributed."""
    import torch.distributed as dist
    rows, cols = grad.shape
    n = rows * cols
    dev = grad.device
    world = dist.get_world_size(group)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    hist = torch.zeros((1, 1), dtype=torch.float32, device=dev)
    scale = torch.ones(1, dtype=torch.float32, device=dev)
    scale_inv = torch.ones(1, dtype=torch.float32, device=dev)
    fp8_amax(grad, amax)
    fp8_scale_update(hist, amax, scale, scale_inv, fmt, margin)
    dist.all_reduce(scale, op=dist.ReduceOp.MIN, group=group)
    shard = fp8_shard_len(n, world)
    q = torch.empty(world * shard, dtype=torch.uint8, device=dev)
    q[n:].zero_()
    fp8_quantize_transpose(grad, scale, fmt, out=q[:n].view(rows, cols))

    def reduce_shard(parts):
        mine = torch.empty(shard, dtype=torch.bfloat16, device=dev)
        fp8_dequant_sum(parts, fmt, scale, mine)
        return mine

    full = fp8_exchange_sum(q, shard, reduce_shard, group)
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    out.view(-1).copy_(full[:n])
    return out
