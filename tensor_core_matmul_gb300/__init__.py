"""bf16 GEMM on GB300 tensor cores (tcgen05 + TMA + TMEM), behind a C ABI.

    C = alpha * A * B + beta * C      A row-major, B and C column-major,
                                      bf16 inputs, fp32 accumulation,
                                      fp32 or bf16 output.
    C = act(alpha * A * B + beta * C + bias)   the fused epilogue (ReLU, GELU)
    gemm_fp8: the same GEMM on 8-bit float operands (E4M3 / E5M2)
    gemm_fp8_ex: A and B in different 8-bit formats; caller workspace
    gemm_fp8_host: 8-bit operands on host buffers
    gemm_quant_i8: int8 codes of act(alpha*A*B + bias) * row_scale + zero_point
    gemm_bf16_layout: A row- or column-major, B column- or row-major
    gemm_bf16_host: the plain GEMM on host buffers (copies in and out included)

The CUDA library (``_lib/libtcgemm.so``, built from ``csrc/``) does all the
work; ``binding`` only marshals arguments.  Build with ``_build.build()``.
"""
from .binding import (OUT_BF16, autotune, autotune_clear, autotune_lookup, OUT_F32, VARIANT_1CTA, VARIANT_1CTA_N64, VARIANT_2CTA, VARIANT_AUTO, TcgemmError,
                      check_device_status, gemm_bf16, gemm_bf16_bias_act, gemm_bf16_host, gemm_bf16_layout, gemm_bf16_raw, gemm_fp8, gemm_fp8_ex, gemm_fp8_host, gemm_quant_i8, gemm_bf16_ws_raw, launch_count, lib, pick_variant,
                      plan, selftest_timeout, tile_order, tile_order_hilbert, version, workspace_bytes)

__all__ = ["OUT_BF16", "autotune", "autotune_clear", "autotune_lookup", "OUT_F32", "VARIANT_1CTA", "VARIANT_1CTA_N64", "VARIANT_2CTA", "VARIANT_AUTO", "TcgemmError",
           "check_device_status", "gemm_bf16", "gemm_bf16_bias_act", "gemm_bf16_host", "gemm_bf16_layout", "gemm_bf16_raw", "gemm_fp8", "gemm_fp8_ex", "gemm_fp8_host", "gemm_quant_i8", "gemm_bf16_ws_raw", "launch_count", "lib", "pick_variant",
           "plan", "selftest_timeout", "tile_order", "tile_order_hilbert", "version", "workspace_bytes"]
