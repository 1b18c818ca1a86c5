"""Keyed error-feedback residuals for weights stored in NVFP4.

[fp4-train] "Usage": an ``ErrorFeedback`` object keeps one fp32 residual per
named weight; ``qdq(key, W, step)`` quantizes W plus that residual to NVFP4,
returns the dequantized bf16 weight and keeps the rounding error for the next
step, so that round-to-nearest no longer stalls on updates below one
quantization step ("Correctness").  ``stochastic=True`` rounds with the
counter-based Philox stream instead (seed, step, element index).

This module is bookkeeping only: every step of the arithmetic runs in the
CUDA library (nvfp4_qdq, whose per-tensor scale comes from its own amax
pass).  The residual of a key is created as zeros on the key's first use,
on the weight's device, and lives until ``reset`` or the object is dropped.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional

import torch

from .codec import nvfp4_qdq


class ErrorFeedback:
    """Error-feedback NVFP4 quantization of named weights.

    ``qdq(key, x, step)`` returns bf16 values q = dequant(quantize(x + r_key))
    and sets r_key <- (x + r_key) - q, all in fp32 inside one fused launch
    pair (amax pass, quantize pass).  ``step(key, w, grad, lr, step)`` applies
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
        for k, v in state.items():
            if v.dtype != torch.float32:
                raise ValueError(f"{k}: residuals are fp32")
        self._res = {k: v for k, v in state.items()}

    # ---------------------------------------------------------------- steps
    def qdq(self, key: str, x: torch.Tensor, step: int = 0) -> torch.Tensor:
        """NVFP4 round trip of x + r_key (x is any float tensor whose size is
        a multiple of 16); returns bf16 values shaped like x."""
        w = x.detach().to(torch.bfloat16).contiguous().clone()
        r = self.residual(key, w)
        nvfp4_qdq(w, None, 0.0, r, rounding=self.rounding, seed=self.seed, step=step,
                  tscale="compute", want_packed=False)
        return w

    def step(self, key: str, w: torch.Tensor, grad: torch.Tensor, lr: float,
             step: int = 0) -> torch.Tensor:
        """W <- qdq((W - lr*G) + r_key) in place on the bf16 weight w (the
        gradient is fp32); returns w."""
        r = self.residual(key, w)
        nvfp4_qdq(w, grad.to(torch.float32).contiguous(), float(lr), r, rounding=self.rounding,
                  seed=self.seed, step=step, tscale="compute", want_packed=False)
        return w

    def qdq_many(self, keys: Iterable[str], xs: Iterable[torch.Tensor],
                 step: int = 0) -> List[torch.Tensor]:
        return [self.qdq(k, x, step) for k, x in zip(keys, xs)]
