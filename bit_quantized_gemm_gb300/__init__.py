"""Exact int8 (W8A8) / W4A8 quantized linear layer for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library libqgemm.so (include/qgemm.h), built by
``bit_quantized_gemm_gb300.build``; this package binds it through ctypes.
"""
from ._lib import (QGError, check_device_error, debug_block_sums, debug_wait_timeout,
                   declared_symbols, gemm_launch_count,
                   gemm_w4a8_mxfp4, gemm_w4a8_q4k, gemm_w8a8_q8_0, linear_w4a8_mxfp4,
                   linear_w4a8_q4k, pack_mxfp4_q8_0,
                   linear_noalloc_scratch_bytes, linear_w8a8_q8_0,
                   linear_w8a8_q8_0_noalloc, linear_workspace_bytes, load, pack_q4k, pack_q8_0,
                   q4k_packed_bytes, q8_0_packed_bytes, quantize_act, quantize_act_static,
                   small_m_max)

__all__ = ["QGError", "check_device_error", "debug_block_sums", "debug_wait_timeout",
           "declared_symbols", "gemm_launch_count",
           "gemm_w4a8_mxfp4", "gemm_w4a8_q4k", "gemm_w8a8_q8_0", "linear_w4a8_mxfp4",
           "linear_w4a8_q4k", "pack_mxfp4_q8_0",
           "linear_noalloc_scratch_bytes", "linear_w8a8_q8_0",
           "linear_w8a8_q8_0_noalloc", "linear_workspace_bytes", "load", "pack_q4k", "pack_q8_0",
           "q4k_packed_bytes", "q8_0_packed_bytes", "quantize_act", "quantize_act_static",
           "small_m_max"]
