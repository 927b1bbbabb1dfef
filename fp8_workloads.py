"""Seeded synthetic inputs for the FP8 linear layer's workloads.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the method's arithmetic: no FP8 encoding, no amax, no scaling,
only random BF16 tensors of the shapes and value distributions below.  Both
the CUDA path and the oracle receive the very same bytes from it.

The workloads stand in for the linear layers of 1B-70B transformers (the
implementation guide's model-size discussion in "Interpreting the results"),
as single layers with synthetic activations, weights and output gradients:

* ``tiny``        M = K = N = 256; X, dY ~ N(0, 1), W ~ N(0, 1) / 16; history 16,
                  margin 0, HYBRID, 4 steps.
* ``sweep``       standalone cast: (2^n / 4096) x 4096 BF16 tensors for
                  n = 16 .. 28, N(0, 1) with 0.1 % of elements multiplied by 100.
* ``mlp7b``       M 8192 tokens, K 4096, N 11008; X ~ N(0, 1), W ~ N(0, 0.02),
                  dY ~ N(0, 1e-3) (standard deviations); history 1024, margin 0.
* ``mlp70b``      M 8192, K 8192, N 28672; X Student-t (3 degrees of freedom)
                  with 1 % of the K input channels multiplied by 50, W ~ N(0, 0.02),
                  dY ~ N(0, 1e-3); history 1024, margin 1.
* ``drift``       M = K = N = 4096; X ~ N(0, 1) * 1.01^t, times 1000 at every step
                  with t % 100 == 50 and all zero at t % 100 == 75; W ~ N(0, 1/64),
                  dY ~ N(0, 1); history 512, margin 0; HYBRID and E4M3-everywhere.

W is drawn once per workload; X and dY are drawn afresh for every step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    x_kind: str          # "normal" | "student_t_outlier_channels" | "drift"
    x_std: float
    w_std: float
    dy_std: float
    history_len: int
    margin: int
    hybrid: bool
    steps: int
    seed: int = 0

    @property
    def flops_per_step(self) -> int:
        """fprop + dgrad + wgrad, 2*M*N*K each."""
        return 6 * self.M * self.N * self.K


WORKLOADS = {
    "tiny": Workload("tiny", 256, 256, 256, "normal", 1.0, 1.0 / 16, 1.0, 16, 0, True, 4),
    "mlp7b": Workload("mlp7b", 8192, 4096, 11008, "normal", 1.0, 0.02, 1e-3, 1024, 0, True, 100),
    "mlp70b": Workload("mlp70b", 8192, 8192, 28672, "student_t_outlier_channels", 1.0, 0.02,
                       1e-3, 1024, 1, True, 50),
    "drift": Workload("drift", 4096, 4096, 4096, "drift", 1.0, 1.0 / 64, 1.0, 512, 0, True, 1000),
}

SWEEP_EXPONENTS = list(range(16, 29))
SWEEP_COLS = 4096


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _seed(base: int, step: int, which: int) -> int:
    return (base * 1_000_003 + step * 101 + which) & 0x7FFF_FFFF_FFFF


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def student_t_bf16(shape, df: int, outlier_frac: float, outlier_mult: float, seed: int,
                   device="cpu") -> torch.Tensor:
    """Student-t(df) as z / sqrt(chi2_df / df); a seeded ``outlier_frac`` of the
    columns (input channels) multiplied by ``outlier_mult``."""
    g = _gen(device, seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(df):
        chi2 += torch.randn(shape, generator=g, device=device, dtype=torch.float32) ** 2
    t = z / torch.sqrt(chi2 / df)
    cols = shape[-1]
    n_out = max(1, int(round(outlier_frac * cols)))
    idx = torch.randperm(cols, generator=g, device=device)[:n_out]
    t[..., idx] *= outlier_mult
    return t.to(torch.bfloat16)


def layer_weight(w: Workload, device="cpu") -> torch.Tensor:
    return normal_bf16((w.N, w.K), w.w_std, _seed(w.seed, 0, 7), device)


def layer_x(w: Workload, step: int, device="cpu") -> torch.Tensor:
    s = _seed(w.seed, step, 1)
    if w.x_kind == "normal":
        return normal_bf16((w.M, w.K), w.x_std, s, device)
    if w.x_kind == "student_t_outlier_channels":
        return student_t_bf16((w.M, w.K), 3, 0.01, 50.0, s, device)
    if w.x_kind == "drift":
        if step % 100 == 75:
            return torch.zeros((w.M, w.K), dtype=torch.bfloat16, device=device)
        g = _gen(device, s)
        x = torch.randn((w.M, w.K), generator=g, device=device, dtype=torch.float32)
        mult = w.x_std * 1.01 ** step * (1000.0 if step % 100 == 50 else 1.0)
        return (x * mult).to(torch.bfloat16)
    raise ValueError(w.x_kind)


def layer_dy(w: Workload, step: int, device="cpu") -> torch.Tensor:
    return normal_bf16((w.M, w.N), w.dy_std, _seed(w.seed, step, 2), device)


def sweep_shape(n: int):
    """Rows x cols of the 2^n-element cast-sweep tensor."""
    total = 1 << n
    return (total // SWEEP_COLS, SWEEP_COLS)


def sweep_tensor(n: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """N(0, 1) with 0.1 % of the elements (seeded positions) multiplied by 100."""
    rows, cols = sweep_shape(n)
    g = _gen(device, _seed(seed, n, 3))
    x = torch.randn(rows * cols, generator=g, device=device, dtype=torch.float32)
    k = max(1, (rows * cols) // 1000)
    pos = torch.randint(0, rows * cols, (k,), generator=g, device=device)
    x[pos] *= 100.0
    return x.to(torch.bfloat16).reshape(rows, cols)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a BF16 tensor's bit patterns (what the oracle takes)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def describe() -> dict:
    return {k: dict(M=v.M, K=v.K, N=v.N, x=v.x_kind, history_len=v.history_len,
                    margin=v.margin, steps=v.steps) for k, v in WORKLOADS.items()}


assert math.isclose(WORKLOADS["tiny"].w_std, 1 / math.sqrt(256))
