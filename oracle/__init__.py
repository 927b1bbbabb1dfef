"""CPU oracle for the FP8 delayed-scaling linear layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package (``python -m oracle`` runs it on its own
and prints its results for a workload's seeded inputs).  The product library never imports,
links or runs it, and it shares no code with the CUDA path: the arithmetic
lives in ``fp8_oracle.c`` (plain C, built here with gcc), and this module only
marshals numpy arrays into it and strings the steps of one training step
together in the order the pages give them.

What each function follows:

* ``quantize`` / ``quantize_f32`` / ``fp8_encode`` / ``fp8_decode`` -- the E4M3 / E5M2 formats of
  "NVIDIA Transformer Engine and FP8 mixed precision: implementation guide",
  section "What are Transformer Engine and FP8 mixed precision", and the
  maxima 448 / 57,344 of the "Definition" table of the "Mixed-precision
  training" wiki note; the Q node of "FP8 quantization with NVIDIA TensorRT".
* ``amax`` / ``amax_f32`` -- dynamic scaling's range monitoring (implementation guide, same
  section) and the Absolute-Max statistic (TensorRT page).
* ``history_update`` -- DelayedScaling's margin / amax_history_len
  (implementation guide, section "Dynamic scaling and the FP8 recipe") with
  the scale formula (fmax / max(history)) / 2^margin.
* ``just_in_time_scale`` -- just-in-time per-tensor scaling (wiki note,
  bullet "per-tensor scaling is the key"): the same formula on this step's
  amax alone.
* ``layernorm`` -- te.LayerNorm's forward (implementation guide, "Basic
  structure of FP8 training code"), in double.
* ``adam_step`` / ``adam_init`` -- Adam (textbook bias correction, AdamW's
  decoupled weight decay) with the optimizer-state precision decoupling of the
  wiki note (first moment FP8, second moment FP16, master weights FP16 with
  tensor scaling), in binary32; the initial state of a weight tensor.
* ``fp8_allreduce`` / ``dequant_sum`` -- FP8 all-reduce with one scale shared
  by all ranks, s'_g = min(s'_1 .. s'_N) (wiki note, bullet "per-tensor
  scaling is the key").
* ``layer_fwd`` / ``layer_bwd`` -- te.Linear inside fp8_autocast with
  Format.HYBRID (E4M3 forward, E5M2 backward; same section) and FP8 GEMMs with
  higher-precision accumulation (wiki note, bullet "extension to FP8").

Every function here is pinned by the ``-m "not gpu"`` tests against values
the pages print, closed forms, library routines or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2 = 0, 1
SLOT_X, SLOT_W, SLOT_Y, SLOT_DY, SLOT_DX = range(5)
N_SLOTS = 5


def build(force: bool = False) -> str:
    """Compile ``fp8_oracle.c`` into ``liboracle.so`` (OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.or_bf16_to_f32.argtypes, lib.or_bf16_to_f32.restype = [ctypes.c_uint16], f32
        lib.or_f32_to_bf16.argtypes, lib.or_f32_to_bf16.restype = [f32], ctypes.c_uint16
        lib.or_fp8_decode.argtypes, lib.or_fp8_decode.restype = [ctypes.c_uint8, ctypes.c_int], ctypes.c_double
        lib.or_fp8_max.argtypes, lib.or_fp8_max.restype = [ctypes.c_int], ctypes.c_double
        lib.or_fp8_encode_f32.argtypes, lib.or_fp8_encode_f32.restype = [f32, ctypes.c_int], ctypes.c_uint8
        lib.or_fp8_encode_f32_array.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.or_fp8_encode_f32_array.restype = None
        lib.or_amax_bf16.argtypes, lib.or_amax_bf16.restype = [vp, i64], f32
        lib.or_quantize.argtypes = [vp, i64, i64, f32, ctypes.c_int, vp, vp]
        lib.or_quantize.restype = None
        lib.or_quantize_f32.argtypes = [vp, i64, f32, ctypes.c_int, vp]
        lib.or_quantize_f32.restype = None
        lib.or_amax_f32.argtypes, lib.or_amax_f32.restype = [vp, i64], f32
        lib.or_history_update.argtypes = [vp, i32, f32, vp, vp, ctypes.c_int, i32]
        lib.or_history_update.restype = None
        lib.or_gemm_tn_f64.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i64, i64, i64, i64, i64, vp]
        lib.or_gemm_tn_f64.restype = None
        lib.or_gemm_tn_exact.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i64, i64, i64, vp]
        lib.or_gemm_tn_exact.restype = ctypes.c_int
        lib.or_epilogue.argtypes = [vp, i64, f32, f32, vp]
        lib.or_epilogue.restype = None
        lib.or_num_threads.argtypes, lib.or_num_threads.restype = [], ctypes.c_int
        lib.or_layernorm.argtypes = [vp, vp, vp, i64, i64, ctypes.c_double, vp, vp, vp]
        lib.or_layernorm.restype = None
        lib.or_f16_decode.argtypes, lib.or_f16_decode.restype = [ctypes.c_uint16], f32
        lib.or_f16_encode.argtypes, lib.or_f16_encode.restype = [f32], ctypes.c_uint16
        lib.or_adam_step.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp] + [f32] * 7 + [i32]
        lib.or_adam_step.restype = None
        lib.or_adam_init.argtypes = [vp, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.or_adam_init.restype = None
        lib.or_dequant_sum.argtypes = [vp, i32, i64, ctypes.c_int, f32, vp]
        lib.or_dequant_sum.restype = None
        _lib_handle = lib
    return _lib_handle


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """Threads the oracle's parallel loops use (OpenMP), 1 without OpenMP."""
    return int(_lib().or_num_threads())


# ----------------------------------------------------------------- formats --

def fp8_decode(code: int, fmt: int) -> float:
    return float(_lib().or_fp8_decode(int(code) & 0xFF, fmt))


def fp8_decode_table(fmt: int) -> np.ndarray:
    """Value of each of the 256 codes (float64; NaN / inf where the format has them)."""
    return np.array([fp8_decode(c, fmt) for c in range(256)], dtype=np.float64)


def fp8_max(fmt: int) -> float:
    return float(_lib().or_fp8_max(fmt))


def fp8_max_f32(fmt: int) -> np.float32:
    return np.float32(fp8_max(fmt))


def fp8_encode(v, fmt: int) -> np.ndarray:
    """Nearest FP8 code of each binary32 value (ties to even code, saturating)."""
    v = _c(np.asarray(v), np.float32).reshape(-1)
    out = np.empty(v.size, dtype=np.uint8)
    _lib().or_fp8_encode_f32_array(v.ctypes.data, v.size, fmt, out.ctypes.data)
    return out


def bf16_to_f32(bits) -> np.ndarray:
    bits = _c(np.asarray(bits), np.uint16)
    f = _lib().or_bf16_to_f32
    return np.array([f(int(b)) for b in bits.reshape(-1)], dtype=np.float32).reshape(bits.shape)


def f32_to_bf16(v) -> np.ndarray:
    v = _c(np.asarray(v), np.float32)
    f = _lib().or_f32_to_bf16
    return np.array([f(float(x)) for x in v.reshape(-1)], dtype=np.uint16).reshape(v.shape)


# ------------------------------------------------------------ the kernels --

def amax(x_bf16: np.ndarray) -> np.float32:
    """max |x| over a BF16 tensor given as its uint16 bit patterns."""
    x = _c(x_bf16, np.uint16)
    return np.float32(_lib().or_amax_bf16(x.ctypes.data, x.size))


def quantize(x_bf16: np.ndarray, scale, fmt: int, transpose: bool = True):
    """Scaled saturating cast of a [rows, cols] BF16 tensor.

    Returns ``(q, q_t)``: FP8 codes [rows, cols] and the transposed copy
    [cols, rows] (``None`` when ``transpose`` is false).
    """
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    qt = np.empty((cols, rows), dtype=np.uint8) if transpose else None
    _lib().or_quantize(x.ctypes.data, rows, cols, float(np.float32(scale)), fmt,
                       q.ctypes.data, qt.ctypes.data if transpose else None)
    return q, qt


def quantize_f32(x: np.ndarray, scale, fmt: int) -> np.ndarray:
    """Scaled saturating cast of an fp32 tensor, element order kept."""
    x = _c(x, np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    _lib().or_quantize_f32(x.ctypes.data, x.size, float(np.float32(scale)), fmt, q.ctypes.data)
    return q


def amax_f32(x: np.ndarray) -> np.float32:
    """max |x| over an fp32 tensor, NaN skipped."""
    x = _c(x, np.float32)
    return np.float32(_lib().or_amax_f32(x.ctypes.data, x.size))


def history_update(hist: np.ndarray, amax_new, scale, scale_inv, fmt: int, margin: int):
    """One delayed-scaling update of one tensor's state; returns new copies."""
    h = np.array(hist, dtype=np.float32, copy=True)
    s = np.array([scale], dtype=np.float32)
    si = np.array([scale_inv], dtype=np.float32)
    _lib().or_history_update(h.ctypes.data, h.size, float(np.float32(amax_new)),
                             s.ctypes.data, si.ctypes.data, fmt, int(margin))
    return h, s[0], si[0]


def gemm_tn(A: np.ndarray, fa: int, B: np.ndarray, fb: int, row0: int = 0,
            nrows: int | None = None) -> np.ndarray:
    """acc[i, j] = sum_k dec(A[row0 + i, k]) * dec(B[j, k]) in double."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    if nrows is None:
        nrows = M - row0
    acc = np.empty((nrows, N), dtype=np.float64)
    _lib().or_gemm_tn_f64(A.ctypes.data, fa, B.ctypes.data, fb, M, N, K, row0, nrows,
                          acc.ctypes.data)
    return acc


def gemm_tn_exact(A: np.ndarray, fa: int, B: np.ndarray, fb: int) -> np.ndarray:
    """Same sum in exact 128-bit integer arithmetic, rounded once to double."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N, _ = B.shape
    acc = np.empty((M, N), dtype=np.float64)
    rc = _lib().or_gemm_tn_exact(A.ctypes.data, fa, B.ctypes.data, fb, M, N, K,
                                 acc.ctypes.data)
    if rc != 0:
        raise ValueError("exact GEMM needs finite FP8 operands")
    return acc


def epilogue(acc: np.ndarray, sa_inv, sb_inv) -> np.ndarray:
    """Dequant to BF16: bf16_rne(fl32(fl32(acc) * fl32(sa_inv * sb_inv)))."""
    a = _c(acc, np.float64)
    y = np.empty(a.shape, dtype=np.uint16)
    _lib().or_epilogue(a.ctypes.data, a.size, float(np.float32(sa_inv)),
                       float(np.float32(sb_inv)), y.ctypes.data)
    return y


# ------------------------------------------------------------- LayerNorm --

def layernorm(x_bf16: np.ndarray, gamma_bf16: np.ndarray, beta_bf16: np.ndarray, eps: float):
    """te.LayerNorm's forward (implementation guide, "Basic structure of FP8
    training code") in double: returns y [rows, cols], mean [rows], rstd [rows]."""
    x = _c(x_bf16, np.uint16)
    g = _c(gamma_bf16, np.uint16)
    b = _c(beta_bf16, np.uint16)
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64)
    mean = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    _lib().or_layernorm(x.ctypes.data, g.ctypes.data, b.ctypes.data, rows, cols, float(eps),
                        y.ctypes.data, mean.ctypes.data, rstd.ctypes.data)
    return y, mean, rstd


# ------------------------------------------------------- FP8 optimizer --

def f16_encode(v) -> np.ndarray:
    """Binary32 -> FP16 codes: nearest value, ties to even, saturating at 65504."""
    v = _c(np.asarray(v), np.float32)
    f = _lib().or_f16_encode
    return np.array([f(float(x)) for x in v.reshape(-1)], dtype=np.uint16).reshape(v.shape)


def f16_decode(h) -> np.ndarray:
    h = _c(np.asarray(h), np.uint16)
    f = _lib().or_f16_decode
    return np.array([f(int(x)) for x in h.reshape(-1)], dtype=np.float32).reshape(h.shape)


@dataclass
class AdamHyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    margin: int = 0

    def bias_corrections(self, t: int):
        """(1 - beta1^t, 1 - beta2^t) as binary32, computed in double."""
        return np.float32(1.0 - self.beta1 ** t), np.float32(1.0 - self.beta2 ** t)


def adam_step(grad_bf16, m1, m1_scale, m1_scale_inv, m2, w16, w_scale, w_scale_inv, hp: AdamHyper,
              t: int):
    """One Adam step on decoupled-precision states (wiki note, bullet
    "precision decoupling"): returns the new (m1, m1_scale, m1_scale_inv, m2,
    w16, w_scale, w_scale_inv, w_bf16, amax[2]) as copies."""
    g = _c(grad_bf16, np.uint16).reshape(-1)
    n = g.size
    m1o = np.array(m1, np.uint8).reshape(-1).copy()
    m2o = np.array(m2, np.uint16).reshape(-1).copy()
    w16o = np.array(w16, np.uint16).reshape(-1).copy()
    wb = np.empty(n, np.uint16)
    sc = np.array([m1_scale, m1_scale_inv, w_scale, w_scale_inv], np.float32)
    am = np.zeros(2, np.float32)
    bc1, bc2 = hp.bias_corrections(t)
    _lib().or_adam_step(g.ctypes.data, n, m1o.ctypes.data, sc[0:].ctypes.data,
                        sc[1:].ctypes.data, m2o.ctypes.data, w16o.ctypes.data,
                        sc[2:].ctypes.data, sc[3:].ctypes.data, wb.ctypes.data, am.ctypes.data,
                        float(np.float32(hp.lr)), float(np.float32(hp.beta1)),
                        float(np.float32(hp.beta2)), float(np.float32(hp.eps)),
                        float(np.float32(hp.weight_decay)), float(bc1), float(bc2), int(hp.margin))
    return m1o, sc[0], sc[1], m2o, w16o, sc[2], sc[3], wb, am


def adam_init(w_bf16, margin: int = 0):
    """Initial decoupled-precision Adam state of a BF16 weight tensor (wiki
    note, bullet "precision decoupling"): zero moments, master weights FP16
    under the just-in-time scale of w (fmax 65504, a history of one).
    Returns (m1, m1_scale, m1_scale_inv, m2, w16, w_scale, w_scale_inv, amax[2])."""
    w = _c(w_bf16, np.uint16).reshape(-1)
    n = w.size
    m1 = np.empty(n, np.uint8)
    m2 = np.empty(n, np.uint16)
    w16 = np.empty(n, np.uint16)
    sc = np.zeros(4, np.float32)
    am = np.zeros(2, np.float32)
    _lib().or_adam_init(w.ctypes.data, n, int(margin), m1.ctypes.data, sc[0:].ctypes.data,
                        sc[1:].ctypes.data, m2.ctypes.data, w16.ctypes.data, sc[2:].ctypes.data,
                        sc[3:].ctypes.data, am.ctypes.data)
    return m1, sc[0], sc[1], m2, w16, sc[2], sc[3], am


# ------------------------------------------------- FP8 all-reduce --

def dequant_sum(parts: np.ndarray, fmt: int, scale) -> np.ndarray:
    """Sum of [nranks, n] FP8 codes sharing one scale, as BF16 bits: the exact
    sum of the decoded codes times fl32(1 / scale), rounded once to BF16."""
    q = _c(parts, np.uint8)
    nranks, n = q.shape
    out = np.empty(n, np.uint16)
    _lib().or_dequant_sum(q.ctypes.data, nranks, n, fmt, float(np.float32(scale)),
                          out.ctypes.data)
    return out


def local_scale(x_bf16: np.ndarray, fmt: int, margin: int) -> np.float32:
    """A rank's own scale for its tensor: the recipe formula on its amax (a
    history of one); 1 when the amax is 0 or not finite."""
    _, s, _ = history_update(np.zeros(1, np.float32), amax(x_bf16), np.float32(1.0),
                             np.float32(1.0), fmt, margin)
    return np.float32(s)


def fp8_allreduce(grads_bf16, fmt: int, margin: int = 0):
    """FP8 all-reduce of per-rank BF16 tensors with the one shared scale
    s'_g = min over ranks of each rank's own scale (wiki note, bullet
    "per-tensor scaling is the key"): every rank casts its tensor with s'_g,
    the FP8 codes are exchanged, and their values are summed and dequantised.
    Returns (BF16 bits of the sum, s'_g, the per-rank codes)."""
    scales = [local_scale(g, fmt, margin) for g in grads_bf16]
    sg = np.float32(min(scales))
    parts = np.stack([quantize(np.asarray(g).reshape(1, -1), sg, fmt, transpose=False)[0][0]
                      for g in grads_bf16])
    return dequant_sum(parts, fmt, sg), sg, parts


# ------------------------------------------------------------- the layer --

@dataclass
class Recipe:
    """DelayedScaling: margin (default 0), amax_history_len (default 1024),
    HYBRID (E4M3 forward, E5M2 backward) or E4M3 everywhere.

    ``current`` selects just-in-time scaling for X, W and dY (the wiki note's
    bullet "per-tensor scaling is the key" names it beside delayed scaling):
    the scale of a tensor comes from its own amax in the same step, through
    the same formula applied to a history of one entry."""
    margin: int = 0
    history_len: int = 1024
    hybrid: bool = True
    current: bool = False

    def formats(self):
        bwd = E5M2 if self.hybrid else E4M3
        return [E4M3, E4M3, E4M3, bwd, bwd]


@dataclass
class State:
    """Per-layer scaling state: 5 slots (X, W, Y, dY, dX)."""
    history: np.ndarray
    amax: np.ndarray = field(default_factory=lambda: np.zeros(N_SLOTS, np.float32))
    scale: np.ndarray = field(default_factory=lambda: np.ones(N_SLOTS, np.float32))
    scale_inv: np.ndarray = field(default_factory=lambda: np.ones(N_SLOTS, np.float32))

    @staticmethod
    def initial(history_len: int) -> "State":
        return State(history=np.zeros((N_SLOTS, history_len), np.float32))

    def copy(self) -> "State":
        return State(self.history.copy(), self.amax.copy(), self.scale.copy(),
                     self.scale_inv.copy())


def just_in_time_scale(st: State, rc: Recipe, slot: int, fmt: int) -> None:
    """Just-in-time scaling of one slot: its scale and inverse from this
    step's amax alone (a history of one), kept when that amax is 0 or inf."""
    _, s, si = history_update(np.zeros(1, np.float32), st.amax[slot], st.scale[slot],
                              st.scale_inv[slot], fmt, rc.margin)
    st.scale[slot], st.scale_inv[slot] = s, si


def layer_fwd(st: State, rc: Recipe, X: np.ndarray, W: np.ndarray, rows=None):
    """Forward of the FP8 linear: Y = X W^T.  ``rows`` (start, count) limits the
    GEMM to a block of Y's rows; the casts always cover the whole tensors."""
    f = rc.formats()
    st.amax[SLOT_X] = amax(X)
    st.amax[SLOT_W] = amax(W)
    if rc.current:
        just_in_time_scale(st, rc, SLOT_X, f[SLOT_X])
        just_in_time_scale(st, rc, SLOT_W, f[SLOT_W])
    X8, X8t = quantize(X, st.scale[SLOT_X], f[SLOT_X])
    W8, W8t = quantize(W, st.scale[SLOT_W], f[SLOT_W])
    r0, nr = rows if rows is not None else (0, X.shape[0])
    acc = gemm_tn(X8, f[SLOT_X], W8, f[SLOT_W], r0, nr)
    Y = epilogue(acc, st.scale_inv[SLOT_X], st.scale_inv[SLOT_W])
    if rows is None:
        st.amax[SLOT_Y] = amax(Y)
    return dict(X8=X8, X8t=X8t, W8=W8, W8t=W8t, Y=Y, Y_acc=acc)


def layer_bwd(st: State, rc: Recipe, dY: np.ndarray, X8t: np.ndarray, W8t: np.ndarray,
              rows=None, wrows=None):
    """Backward: dX = dY W (dgrad) and dW = dY^T X (wgrad), FP8 operands.
    ``rows`` limits dgrad to a block of dX's rows, ``wrows`` wgrad to a block
    of dW's rows; the cast always covers the whole of dY."""
    f = rc.formats()
    st.amax[SLOT_DY] = amax(dY)
    if rc.current:
        just_in_time_scale(st, rc, SLOT_DY, f[SLOT_DY])
    dY8, dY8t = quantize(dY, st.scale[SLOT_DY], f[SLOT_DY])
    r0, nr = rows if rows is not None else (0, dY.shape[0])
    acc_dx = gemm_tn(dY8, f[SLOT_DY], W8t, f[SLOT_W], r0, nr)
    dX = epilogue(acc_dx, st.scale_inv[SLOT_DY], st.scale_inv[SLOT_W])
    if rows is None:
        st.amax[SLOT_DX] = amax(dX)
    wr0, wnr = wrows if wrows is not None else (0, dY.shape[1])
    acc_dw = gemm_tn(dY8t, f[SLOT_DY], X8t, f[SLOT_X], wr0, wnr)
    dW = epilogue(acc_dw, st.scale_inv[SLOT_DY], st.scale_inv[SLOT_X])
    return dict(dY8=dY8, dY8t=dY8t, dX=dX, dX_acc=acc_dx, dW=dW, dW_acc=acc_dw)


def layer_update(st: State, rc: Recipe) -> None:
    """Delayed-scaling update of all five slots, after forward and backward."""
    f = rc.formats()
    for t in range(N_SLOTS):
        h, s, si = history_update(st.history[t], st.amax[t], st.scale[t], st.scale_inv[t],
                                  f[t], rc.margin)
        st.history[t], st.scale[t], st.scale_inv[t] = h, s, si
