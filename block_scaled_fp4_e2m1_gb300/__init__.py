"""Block-scaled FP4 (E2M1) codec for GB300 (sm_103a).

The compute path is the CUDA library ``libfp4codec.so`` (C ABI in
include/fp4codec.h); this package is its Python binding.  Importing the
package does not load the library; the first call does, and raises if it has
not been built (there is no CPU fallback).
"""
from .codec import (Batch, Segments, fp4_blocked_scales_size, fp4_scaled_dequantize,
                    fp4_scaled_dequantize_dev, fp4_scaled_quantize, fp4_scaled_quantize_amax, fp4_scales_from_blocked, fp4_scales_to_blocked,
                    fp4_seg_scale_offsets, fp4_to_fp8_col, fp4_to_fp8_row,
                    fp4quant_decode, fp4quant_encode, fp8_to_fp4_row, kernel_launches,
                    wait_timeouts,
                    mxfp4_dequantize, mxfp4_quantize, nvfp4_amax, nvfp4_amax_batched,
                    nvfp4_dequantize, nvfp4_dequantize_batched, nvfp4_qdq, nvfp4_qdq_amax,
                    nvfp4_quantize, nvfp4_quantize_batched, nvfp4_quantize_batched_blocked,
                    nvfp4_quantize_blocked,
                    nvfp4_quantize_noalloc)
from .error_feedback import ErrorFeedback
from .quality import fp4_quality

__all__ = [
    "Batch", "ErrorFeedback", "Segments", "fp4_blocked_scales_size", "fp4_quality",
    "fp4_scaled_dequantize", "fp4_scaled_dequantize_dev", "fp4_scaled_quantize",
    "fp4_scaled_quantize_amax", "fp4_scales_from_blocked",
    "fp4_scales_to_blocked", "fp4_seg_scale_offsets", "fp4_to_fp8_col", "fp4_to_fp8_row",
    "fp4quant_decode", "fp4quant_encode", "fp8_to_fp4_row", "kernel_launches",
    "wait_timeouts",
    "mxfp4_dequantize", "mxfp4_quantize", "nvfp4_amax", "nvfp4_amax_batched",
    "nvfp4_dequantize", "nvfp4_dequantize_batched", "nvfp4_qdq", "nvfp4_qdq_amax",
    "nvfp4_quantize", "nvfp4_quantize_batched", "nvfp4_quantize_batched_blocked",
    "nvfp4_quantize_blocked",
    "nvfp4_quantize_noalloc",
]
