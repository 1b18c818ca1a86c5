"""Keyed error-feedback residuals for weights stored in NVFP4.

[fp4-train] "Usage": an ``ErrorFeedback`` object keeps one fp32 residual per
named weight; ``qdq(key, W, step)`` quantizes W plus that residual to NVFP4,
returns the dequantized bf16 weight and keeps the rounding error for the next
step, so that round-to-nearest no longer stalls on updates below one
quantization step ("Correctness").  ``stochastic=True`` rounds with the
counter-based Philox stream instead (seed, step, element index).

This module is bookkeeping only: every step of the arithmetic runs in the
CUDA library.  A bf16 input goes through nvfp4_qdq (amax pass, then the fused
quantize and dequantize in place on a bf16 copy); an fp32 input goes through
nvfp4_quantize with the residual (amax pass, quantize) and nvfp4_dequantize
to bf16, so that the input is never rounded before the residual is added.
Both give v = x + r in fp32, q = dequant(quantize(v)) in fp32, r <- v - q,
and return bf16(q).  The residual of a key is created as zeros on the key's
first use, on the input's device, and lives until ``reset`` or the object is
dropped.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional

import torch

from .codec import nvfp4_dequantize, nvfp4_qdq, nvfp4_quantize


class ErrorFeedback:
    """Error-feedback NVFP4 quantization of named weights.

    ``qdq(key, x, step)`` returns bf16 values bf16(q), q = dequant(quantize(v))
    with v = x + r_key, and sets r_key <- v - q, all in fp32: x, as given
    (bf16, fp16 or fp32; fp16 widens exactly), is added to the residual
    before anything is rounded.  ``step(key, w, grad, lr, step)`` applies
    the update W <- qdq((W - lr*G) + r) in place on a bf16 weight, with the
    subtraction fused into the kernel.
    """

    def __init__(self, stochastic: bool = False, seed: int = 0):
        self.rounding = "sr" if stochastic else "rtn"
        self.seed = int(seed)
        self._res: Dict[str, torch.Tensor] = {}

    # ------------------------------------------------------------ residuals
    def residual(self, key: str, like: torch.Tensor) -> torch.Tensor:
        """The fp32 residual of `key`, created as zeros shaped like `like`."""
        r = self._res.get(key)
        if r is None:
            r = torch.zeros(like.shape, dtype=torch.float32, device=like.device)
            self._res[key] = r
        elif r.shape != like.shape or r.device != like.device:
            raise ValueError(f"{key}: residual is {tuple(r.shape)} on {r.device}, "
                             f"weight is {tuple(like.shape)} on {like.device}")
        return r

    def keys(self) -> List[str]:
        return list(self._res)

    def reset(self, key: Optional[str] = None) -> None:
        """Forget one residual, or all of them."""
        if key is None:
            self._res.clear()
        else:
            self._res.pop(key, None)

    def state_dict(self) -> Dict[str, torch.Tensor]:
        return {k: v for k, v in self._res.items()}

    def load_state_dict(self, state: Dict[str, torch.Tensor]) -> None:
        """Replace every residual; each must be an fp32 tensor.  A residual
        is stored contiguous (the kernels read it as a flat array)."""
        for k, v in state.items():
            if not isinstance(v, torch.Tensor) or v.dtype != torch.float32:
                raise ValueError(f"{k}: residuals are fp32 tensors")
        self._res = {k: v.detach().contiguous() for k, v in state.items()}

    # ---------------------------------------------------------------- steps
    def qdq(self, key: str, x: torch.Tensor, step: int = 0) -> torch.Tensor:
        """NVFP4 round trip of x + r_key; x is a bf16, fp16 or fp32 CUDA tensor
        whose size is a multiple of 16.  Returns bf16 values shaped like x."""
        x = x.detach()
        if x.dtype == torch.bfloat16:
            w = x.contiguous().clone()
            r = self.residual(key, w)
            nvfp4_qdq(w.view(-1), None, 0.0, r.view(-1), rounding=self.rounding,
                      seed=self.seed, step=step, tscale="compute", want_packed=False)
            return w
        if x.dtype == torch.float16:
            x = x.to(torch.float32)  # exact
        if x.dtype != torch.float32:
            raise ValueError(f"{key}: x must be bfloat16, float16 or float32, got {x.dtype}")
        x = x.contiguous()
        r = self.residual(key, x)
        packed, scales, ts = nvfp4_quantize(x.view(-1), residual=r.view(-1),
                                            rounding=self.rounding, seed=self.seed, step=step,
                                            tscale="compute")
        return nvfp4_dequantize(packed, scales, ts, x.shape, torch.bfloat16)

    def step(self, key: str, w: torch.Tensor, grad: torch.Tensor, lr: float,
             step: int = 0) -> torch.Tensor:
        """W <- qdq((W - lr*G) + r_key) in place on the bf16 weight w; the
        gradient is fp32 (or is widened to it) with w's number of elements, on
        w's device.  Returns w."""
        if not w.is_contiguous() or w.dtype != torch.bfloat16:
            raise ValueError(f"{key}: w must be a contiguous bfloat16 tensor")
        if grad.numel() != w.numel():
            raise ValueError(f"{key}: grad has {grad.numel()} elements, w has {w.numel()}")
        if grad.device != w.device:
            raise ValueError(f"{key}: grad is on {grad.device}, w on {w.device}")
        r = self.residual(key, w)
        nvfp4_qdq(w.view(-1), grad.detach().to(torch.float32).contiguous().view(-1), float(lr),
                  r.view(-1), rounding=self.rounding, seed=self.seed, step=step,
                  tscale="compute", want_packed=False)
        return w

    def qdq_many(self, keys: Iterable[str], xs: Iterable[torch.Tensor],
                 step: int = 0) -> List[torch.Tensor]:
        return [self.qdq(k, x, step) for k, x in zip(keys, xs)]
