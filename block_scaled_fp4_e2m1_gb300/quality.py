"""Quantization quality of a weight matrix, the four ways of [WP2]'s table
("Block scaling"): rounding straight to FP4, one scale per matrix, MXFP4 (32
per block, power-of-two scales) and NVFP4 (16 per block, e4m3 scales under
a per-tensor fp32 scale).

For each it reports the share of weights whose stored value is 0 and the
average error, which the page defines as the average distance between a
weight and its stored value divided by the average size of a weight.  The
four round trips run in the CUDA library; the two statistics are plain
float64 reductions over its outputs.
"""
from __future__ import annotations

import math
from typing import Dict

import torch

from .codec import (fp4_scaled_dequantize, fp4_scaled_dequantize_dev, fp4_scaled_quantize,
                    fp4_scaled_quantize_amax, mxfp4_dequantize, mxfp4_quantize, nvfp4_amax,
                    nvfp4_dequantize, nvfp4_quantize)

METHODS = ("straight", "per_matrix", "mxfp4", "nvfp4")


def round_trips(w: torch.Tensor) -> Dict[str, torch.Tensor]:
    """The stored (dequantized) fp32 values of w [rows, cols] under each
    method; cols % 32 == 0."""
    rows, cols = w.shape
    x = w.contiguous().view(-1)
    n = x.numel()
    amax = nvfp4_amax(x)
    if not math.isfinite(float(amax.item())):
        raise ValueError("the matrix holds a non-finite value")
    pk, s = fp4_scaled_quantize_amax(x, amax)  # s = RN(amax / 6), on the device
    out = {
        "straight": fp4_scaled_dequantize(fp4_scaled_quantize(x, 1.0), n, 1.0),
        "per_matrix": fp4_scaled_dequantize_dev(pk, n, s),
    }
    pk, sc = mxfp4_quantize(w.contiguous())
    out["mxfp4"] = mxfp4_dequantize(pk, sc, torch.float32).view(-1)
    pk, sc, ts = nvfp4_quantize(x)
    out["nvfp4"] = nvfp4_dequantize(pk, sc, ts, (n,), torch.float32)
    return out


def stats(w: torch.Tensor, q: torch.Tensor) -> Dict[str, float]:
    """zero: share of weights stored as 0; error: sum |w - q| / sum |w|."""
    x = w.reshape(-1).to(torch.float64)
    q = q.reshape(-1).to(torch.float64)
    return {"zero": int((q == 0).sum()) / q.numel(),
            "error": float((x - q).abs().sum() / x.abs().sum())}


def fp4_quality(w: torch.Tensor) -> Dict[str, Dict[str, float]]:
    """{method: {"zero": ..., "error": ...}} for the bf16 or fp32 matrix w."""
    return {m: stats(w, q) for m, q in round_trips(w).items()}
