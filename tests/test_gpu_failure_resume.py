"""Failure detection and checkpoint/resume on the GPU.

* A bounded wait that runs out (a barrier nothing ever signals, through the
  library's own wait) is reported by fp8_sync_status as FP8_ERR_TIMEOUT once,
  the flag clears, and the context keeps computing correct results.  No
  fault, trap or unbounded wait is involved.
* The scaling state is the whole state of delayed scaling (the guide's
  recipe section keeps it in state_dict): saving it after k steps and
  restoring it into a fresh layer must continue bit-identically to an
  uninterrupted run -- histories, scales and the step's outputs."""
import numpy as np
import pytest
import torch

import fp8_workloads as wl
import oracle as o
from helpers import assert_gemm_close, host_bf16_bits

pytestmark = pytest.mark.gpu

FP8_ERR_TIMEOUT = 4


def test_bounded_wait_reports_timeout_and_context_survives():
    import fp8_mixed_precision_amax_gb300 as f
    f.fp8_sync_status()
    f.fp8_selftest_wait_timeout(100_000_000)            # gives up after 0.1 s
    with pytest.raises(f.Fp8Error) as e:
        f.fp8_sync_status()
    assert e.value.status == FP8_ERR_TIMEOUT
    f.fp8_sync_status()                                 # reported once, then clear
    with pytest.raises(f.Fp8Error):
        f.fp8_selftest_wait_timeout(0)                  # rejected on the host
    # the context still computes: a GEMM against the oracle
    g = torch.Generator().manual_seed(3)
    A = o.fp8_encode((torch.randn(384, 512, generator=g) * 2).numpy(), o.E4M3).reshape(384, 512)
    B = o.fp8_encode(torch.randn(256, 512, generator=g).numpy(), o.E4M3).reshape(256, 512)
    D = torch.empty((384, 256), dtype=torch.bfloat16, device="cuda")
    one = torch.ones(1, device="cuda")
    f.fp8_gemm_tn(torch.from_numpy(A).cuda(), o.E4M3, torch.from_numpy(B).cuda(), o.E4M3, one, one,
                  D)
    f.fp8_sync_status()
    assert_gemm_close(host_bf16_bits(D), o.epilogue(o.gemm_tn(A, o.E4M3, B, o.E4M3), 1.0, 1.0),
                      512, "after timeout")


def test_checkpoint_resume_is_bit_identical():
    import fp8_mixed_precision_amax_gb300 as f
    w = wl.Workload("resume", 512, 1024, 768, "normal", 1.0, 0.02, 1e-3, 16, 0, True, 6)
    W = wl.layer_weight(w, "cuda")
    rc = f.Recipe(w.margin, w.history_len, w.hybrid)
    X = [wl.layer_x(w, t, "cuda") for t in range(6)]
    dY = [wl.layer_dy(w, t, "cuda") for t in range(6)]
    full = f.Fp8Linear(W, w.M, rc)
    for t in range(6):
        full.step(X[t], dY[t])
    first = f.Fp8Linear(W, w.M, rc)
    for t in range(3):
        first.step(X[t], dY[t])
    saved = {k: v.detach().cpu().clone() for k, v in first.meta.state_dict().items()}
    resumed = f.Fp8Linear(W, w.M, rc)
    resumed.meta.load_state_dict(saved)
    for t in range(3, 6):
        resumed.step(X[t], dY[t])
    torch.cuda.synchronize()
    for k, v in full.meta.state_dict().items():
        a = v.detach().cpu().numpy()
        b = resumed.meta.state_dict()[k].detach().cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), k
    for name in ("Y", "dX", "dW"):
        assert np.array_equal(host_bf16_bits(getattr(full, name)),
                              host_bf16_bits(getattr(resumed, name))), name
    f.fp8_sync_status()
