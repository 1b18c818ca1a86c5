"""Seeded synthetic inputs for the five workloads (shapes and distributions of
the pages' workloads).  This module holds no quantization arithmetic: it only
draws random tensors, so both the CUDA path and the CPU oracle can be fed the
same bytes.

Every generator takes a ``device`` and draws from a ``torch.Generator`` on it,
seeded explicitly; the same (seed, device, shape) always gives the same bytes.

Workloads:
  nvfp4_roundtrip   fp32 [1024, 1024] ~ N(0, 0.02), 0.1% entries ~ N(0, 1)
  fp4quant_acts     bf16 [16384, 4096] Student-t(df=4), 8 fixed channels x20
  nvfp4_train       bf16 W [6144, 2048] ~ N(0, 0.02); per step G ~ N(0, 1)
  moe_tokens        bf16 [32768, 7168] ~ N(0, 1), top-8 of 256 experts with
                    Zipf(s=1.1) expert popularity, rows sorted by expert
  qwen3_8b_weights  36 layers of q/o 4096x4096, k/v 1024x4096, gate/up
                    12288x4096, down 4096x12288, bf16 Laplace(median |w| =
                    0.017) with 16 outliers |w| in [0.3, 1.2] (max 1.2)
"""
from __future__ import annotations

import math

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def nvfp4_roundtrip(seed: int = 0, shape=(1024, 1024), device="cpu") -> torch.Tensor:
    """fp32 N(0, 0.02) with round(0.001 n) seeded positions replaced by N(0, 1)."""
    g = _gen(seed, device)
    n = shape[0] * shape[1]
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32) * 0.02
    k = int(round(0.001 * n))
    pos = torch.randperm(n, generator=g, device=device)[:k]
    x[pos] = torch.randn(k, generator=g, device=device, dtype=torch.float32)
    return x.view(shape)


def fp4quant_acts(seed: int = 0, tokens: int = 16384, hidden: int = 4096,
                  device="cpu") -> torch.Tensor:
    """bf16 Student-t(df=4) activations; 8 seeded channels (the same for all
    tokens) multiplied by 20."""
    g = _gen(seed, device)
    z = torch.randn(tokens, hidden, generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros_like(z)
    for _ in range(4):
        chi += torch.randn(tokens, hidden, generator=g, device=device, dtype=torch.float32) ** 2
    t = z / torch.sqrt(chi / 4.0)
    ch = torch.randperm(hidden, generator=g, device=device)[:8]
    t[:, ch] *= 20.0
    return t.to(torch.bfloat16)


def nvfp4_train_weight(seed: int = 0, shape=(6144, 2048), device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    w = torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16)


def nvfp4_train_grad(seed: int, step: int, shape=(6144, 2048), device="cpu") -> torch.Tensor:
    """G_t ~ N(0, 1), fp32, from seed + 1 + t."""
    g = _gen(seed + 1 + step, device)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def moe_tokens(seed: int = 0, tokens: int = 32768, hidden: int = 7168,
               device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn(tokens, hidden, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def moe_routing(seed: int = 0, tokens: int = 32768, experts: int = 256, topk: int = 8,
                zipf_s: float = 1.1):
    """Top-k routing with Zipf(s) expert popularity over a seeded permutation
    of the experts.  Returns (row_token int64[tokens*topk], row_off
    int64[experts+1]): dispatched row i holds token row_token[i]; rows are
    grouped by expert (expert e owns rows row_off[e] .. row_off[e+1]-1) and
    ordered by token inside a group.  Always drawn on the CPU."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(experts, generator=g)
    rank = torch.empty(experts, dtype=torch.float64)
    rank[perm] = torch.arange(1, experts + 1, dtype=torch.float64)
    w = rank ** (-zipf_s)
    choice = torch.multinomial(w.expand(tokens, experts), topk, replacement=False,
                               generator=g)                     # [tokens, topk]
    expert = choice.reshape(-1)
    token = torch.arange(tokens).repeat_interleave(topk)
    key = expert * tokens + token                               # sort by expert, then token
    order = torch.argsort(key)
    row_token = token[order].contiguous()
    counts = torch.bincount(expert, minlength=experts)
    row_off = torch.zeros(experts + 1, dtype=torch.int64)
    row_off[1:] = torch.cumsum(counts, 0)
    return row_token, row_off


def qwen3_8b_weight_shapes(layers: int = 36):
    """[(rows, cols)] of the 7 projection matrices of each layer."""
    per_layer = [(4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096),   # q, k, v, o
                 (12288, 4096), (12288, 4096), (4096, 12288)]              # gate, up, down
    return per_layer * layers


def laplace_weight(seed: int, shape, median_abs: float = 0.017, outliers: int = 16,
                   max_abs: float = 1.2, device="cpu") -> torch.Tensor:
    """bf16 Laplace(0, b) with median |w| = median_abs (b = median / ln 2), and
    ``outliers`` seeded entries with |w| ~ U(0.3, max_abs), one of them exactly
    +-max_abs."""
    g = _gen(seed, device)
    n = shape[0] * shape[1]
    b = median_abs / math.log(2.0)
    # rand() can return exactly 0; keep |u| < 1/2 so that every weight is finite
    u = torch.rand(n, generator=g, device=device, dtype=torch.float32).clamp_(min=2.0 ** -25) - 0.5
    w = -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    if n <= 2 ** 31 - 1:
        pos = torch.randperm(n, generator=g, device=device)[:outliers]
    else:  # randperm's sort stops at 2^31 elements: one position per stratum
        span = n // outliers
        pos = (torch.randint(0, span, (outliers,), generator=g, device=device) +
               span * torch.arange(outliers, device=device))
    mag = 0.3 + (max_abs - 0.3) * torch.rand(outliers, generator=g, device=device)
    mag[0] = max_abs
    sgn = torch.where(torch.rand(outliers, generator=g, device=device) < 0.5, -1.0, 1.0)
    w[pos] = mag * sgn
    return w.view(shape).to(torch.bfloat16)


def size_sweep_bytes():
    """1 MiB .. 4 GiB of bf16 in powers of two, each shaped [-1, 4096]."""
    return [1 << k for k in range(20, 33)]
