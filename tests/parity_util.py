"""Helpers for the GPU parity tests: move tensors between the CUDA path and
the CPU oracle, and compare bit patterns."""
import numpy as np
import torch

import oracle as ora


def ensure_built():
    from block_scaled_fp4_e2m1_gb300 import build as b
    b.build()
    ora.build()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f32_np(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a float32 or bfloat16 tensor."""
    if t.dtype == torch.bfloat16:
        return ora.bf16_to_f32(bf16_bits(t))
    return t.detach().contiguous().cpu().numpy().astype(np.float32, copy=False)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bits_equal(got, want, what=""):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    if got.dtype == np.float32:
        got, want = f32_bits(got), f32_bits(want)
    bad = np.nonzero(got.ravel() != want.ravel())[0]
    if bad.size:
        i = bad[:8]
        raise AssertionError(f"{what}: {bad.size} of {got.size} differ; first at {i.tolist()}: "
                             f"got {got.ravel()[i].tolist()} want {want.ravel()[i].tolist()}")


def dev():
    return torch.device("cuda", 0)
