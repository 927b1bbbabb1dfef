"""The code tables the full-size GPU layer checks use (CPU only): the
oracle's cast of every BF16 bit pattern at one scale, indexed by a tensor's
bits, is the oracle's cast of that tensor."""
import numpy as np
import torch

import oracle as o
from helpers import assert_fp8_equal, host_bf16_bits, oracle_code_table


def test_oracle_code_table_is_the_oracle_cast():
    """The code table the full-size checks use is the oracle's cast itself:
    on a seeded tensor, table[x_bits] and its transpose equal o.quantize's
    codes and transposed copy, both formats, several scales (CPU side)."""
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(96, 160, generator=g) * 7.0).to(torch.bfloat16)
    x[0, :4] = torch.tensor([float("inf"), -float("inf"), float("nan"), 0.0])
    xb = host_bf16_bits(x)
    for fmt in (o.E4M3, o.E5M2):
        for s in (1.0, 37.5, 2.0 ** -20, 3.0e9):
            t = oracle_code_table(s, fmt)
            q, qt = o.quantize(xb, np.float32(s), fmt)
            assert_fp8_equal(t[xb], q, fmt, "rows")
            assert_fp8_equal(np.ascontiguousarray(t[xb].T), qt, fmt, "transposed")
