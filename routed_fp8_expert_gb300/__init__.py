"""Routed FP8 Mixture-of-Experts FFN forward for GB300 (sm_103a).

The compute lives in libmoe_fp8.so (hand-written CUDA, C ABI in
include/moe_fp8.h); this package is its ctypes binding. Build the library
with ``routed_fp8_expert_gb300.build.build()``.
"""
from ._lib import (MOE_ERR_ARG, MOE_ERR_CUDA, MOE_ERR_INDEX, MOE_ERR_TIMEOUT, MOE_ERR_UNSUPPORTED, MOE_OK,  # noqa: F401
                   RMS_NORM_EPS, MoeCfg, MoeError, block_ffn_forward, cfg_of, check_device_error, combine, combine_residual_rmsnorm,
                   dense_swiglu_fp8, dense_workspace, expert_down_fp8, expert_gateup_fp8, expert_gemm_fp8,
                   last_launch_count, layer_forward, load, pack_weights_fp8, permute, permute_noalloc, permuted_rows, quant_fp8_1x128, quant_permute_fp8,
                   rmsnorm_quant_fp8, route, test_wait_timeout, workspace, workspace_bytes)
