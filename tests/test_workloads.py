"""The seeded input generators: determinism, shapes and value distributions."""
import numpy as np
import torch

import fp8_workloads as wl


def test_seeded_and_deterministic():
    w = wl.WORKLOADS["tiny"]
    a, b = wl.layer_x(w, 3), wl.layer_x(w, 3)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(wl.layer_x(w, 4).view(torch.int16), a.view(torch.int16))
    assert wl.layer_weight(w).shape == (w.N, w.K) and a.dtype == torch.bfloat16
    assert wl.layer_dy(w, 0).shape == (w.M, w.N)


def test_distributions():
    w = wl.WORKLOADS["tiny"]
    assert abs(wl.layer_weight(w).float().std().item() - 1 / 16) < 0.003
    d = wl.WORKLOADS["drift"]
    small = wl.Workload("d", 64, 256, 64, "drift", 1.0, 1 / 64, 1.0, 512, 0, True, 1000)
    s0 = wl.layer_x(small, 1).float().std().item()
    s50 = wl.layer_x(small, 50).float().std().item()
    assert 500 < s50 / s0 < 2000
    assert wl.layer_x(small, 75).abs().max().item() == 0
    t = wl.student_t_bf16((512, 200), 3, 0.01, 50.0, seed=1).float()
    colmax = t.abs().max(dim=0).values
    assert (colmax > 200).sum().item() >= 2     # the two outlier channels
    assert d.flops_per_step == 6 * 4096 ** 3


def test_sweep_outliers():
    x = wl.sweep_tensor(16).float()
    assert x.shape == (16, 4096)
    frac = (x.abs() > 10).float().mean().item()
    assert 0.0005 < frac < 0.0015
