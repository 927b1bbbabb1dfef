"""GB300-native FP8 mixed-precision linear layer with per-tensor delayed scaling.

The compute lives in ``libfp8amax.so`` (hand-written sm_103a kernels behind the
C ABI of ``include/fp8amax.h``); this package is its Python binding.  Importing
it loads the library and fails if it has not been built (``build.build()``).
"""
from .api import (AdamHyper, E4M3, E5M2, NUM_SLOTS, SLOT_DX, SLOT_DY, SLOT_W, SLOT_X, SLOT_Y,
                  Fp8AdamState, Fp8Error, Fp8LayerNormLinear, Fp8Linear, Meta, Recipe,
                  allreduce_amax, fp8_allreduce, fp8_amax, fp8_amax_scale_update,
                  fp8_dequant_sum, fp8_exchange_sum, fp8_gemm_tn, fp8_gemm_tn_grouped,
                  fp8_layernorm_linear_fwd, fp8_layernorm_quantize_transpose,
                  fp8_layernorm_stats, fp8_linear_bwd,
                  fp8_linear_bwd_noalloc, fp8_linear_fwd, fp8_quantize_f32,
                  fp8_quantize_transpose, fp8_quantize_transpose_current,
                  fp8_quantize_transpose_grouped, fp8_scale_update, fp8_selftest_wait_timeout,
                  fp8_set_clock_probe, fp8_shard_len, fp8_sync_status, header_functions, library)

__all__ = [n for n in dir() if not n.startswith("_")]
