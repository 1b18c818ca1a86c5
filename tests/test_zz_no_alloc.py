"""GPU test of nvfp4_quantize_noalloc, the entry point for callers that
cannot allocate device memory (a plugin handed only its tensors by a host
framework that owns all device memory, or C code without a device
allocator): it must give exactly what nvfp4_quantize in COMPUTE mode gives
with a caller-supplied workspace, on two calls in a row (the second reuses
the library's workspace slot, which each call clears).

The file is named to be collected last, so a run that stops at the first
failure has run every other test before this one."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _lib():
    from block_scaled_fp4_e2m1_gb300 import build as b
    b.build()
    from block_scaled_fp4_e2m1_gb300 import _lib as L
    return L


def _call_noalloc(L, x, residual, rounding, seed, step):
    n = x.numel()
    dev = x.device
    ts = torch.full((1,), -3.0, dtype=torch.float32, device=dev)
    packed = torch.empty(n // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(n // 16, dtype=torch.uint8, device=dev)
    dt = 1 if x.dtype == torch.bfloat16 else 0
    st = L.lib().nvfp4_quantize_noalloc(
        x.data_ptr(), dt, n, None if residual is None else residual.data_ptr(), rounding, seed,
        step, ts.data_ptr(), packed.data_ptr(), scales.data_ptr(),
        torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, L.lib().fp4_status_string(st)
    return packed, scales, ts


def _call_existing(L, x, residual, rounding, seed, step):
    n = x.numel()
    dev = x.device
    ts = torch.full((1,), -3.0, dtype=torch.float32, device=dev)
    ws = torch.full((1,), 123.0, dtype=torch.float32, device=dev)
    packed = torch.empty(n // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(n // 16, dtype=torch.uint8, device=dev)
    dt = 1 if x.dtype == torch.bfloat16 else 0
    st = L.lib().nvfp4_quantize(
        x.data_ptr(), dt, n, None if residual is None else residual.data_ptr(), rounding, seed,
        step, 1, ts.data_ptr(), ws.data_ptr(), packed.data_ptr(), scales.data_ptr(),
        torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, L.lib().fp4_status_string(st)
    return packed, scales, ts


def _same(a, b, what):
    assert torch.equal(a.cpu(), b.cpu()), what


@pytest.mark.parametrize("dtype,rounding", [(torch.bfloat16, 0), (torch.float32, 1)])
def test_noalloc_matches_existing_entry_point_twice(dtype, rounding):
    L = _lib()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cpu").manual_seed(17)
    # the second tensor has a smaller amax than the first: a slot left
    # uncleared by the first call would give it the wrong tensor scale
    xs = [(torch.randn(16 * 5000, generator=g) * 3.0).to(dtype).to(dev),
          (torch.randn(16 * 3001, generator=g) * 0.01).to(dtype).to(dev)]
    for i, x in enumerate(xs):
        got = _call_noalloc(L, x, None, rounding, 9, i)
        want = _call_existing(L, x, None, rounding, 9, i)
        torch.cuda.synchronize()
        _same(got[2], want[2], f"tensor scale, call {i}")
        _same(got[0], want[0], f"packed, call {i}")
        _same(got[1], want[1], f"scales, call {i}")
        assert got[2].item() > 0


def test_noalloc_with_residual_twice():
    L = _lib()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cpu").manual_seed(5)
    x = (torch.randn(16 * 2048, generator=g) * 0.02).to(dev)
    r_a = (torch.randn(x.numel(), generator=g) * 1e-3).to(dev)
    r_b = r_a.clone()
    for step in range(2):
        got = _call_noalloc(L, x, r_a, 1, 3, step)
        want = _call_existing(L, x, r_b, 1, 3, step)
        torch.cuda.synchronize()
        _same(got[2], want[2], f"tensor scale, step {step}")
        _same(got[0], want[0], f"packed, step {step}")
        _same(got[1], want[1], f"scales, step {step}")
        _same(r_a, r_b, f"residual, step {step}")


def test_noalloc_argument_checks():
    L = _lib()
    A = 0x100000
    f = L.lib().nvfp4_quantize_noalloc
    assert f(A, 1, 15, None, 0, 0, 0, A, A, A, None) == 3      # n % 16
    assert f(A, 1, 16, None, 0, 0, 0, None, A, A, None) == 1   # tensor_scale
    assert f(A + 8, 1, 16, None, 0, 0, 0, A, A, A, None) == 2  # x alignment
    assert f(A, 9, 16, None, 0, 0, 0, A, A, A, None) == 4      # dtype


def test_noalloc_empty_tensor_publishes_scale_one():
    """n = 0: nothing to quantize, but the tensor scale is still written
    (amax 0 gives scale 1), as nvfp4_quantize does in COMPUTE mode."""
    L = _lib()
    dev = torch.device("cuda", 0)
    for dtype in (torch.bfloat16, torch.float32):
        x = torch.empty(0, dtype=dtype, device=dev)
        _, _, ts = _call_noalloc(L, x, None, 0, 0, 0)
        _, _, ts_want = _call_existing(L, x, None, 0, 0, 0)
        torch.cuda.synchronize()
        assert ts.item() == 1.0 and ts_want.item() == 1.0


def test_noalloc_allocates_nothing():
    """Warmed-up calls leave the device's free memory and PyTorch's
    allocator exactly as they were."""
    L = _lib()
    dev = torch.device("cuda", 0)
    x = (torch.randn(16 * 4096, generator=torch.Generator().manual_seed(3)) * 0.1).to(dev)
    n = x.numel()
    ts = torch.empty(1, dtype=torch.float32, device=dev)
    packed = torch.empty(n // 2, dtype=torch.uint8, device=dev)
    scales = torch.empty(n // 16, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call():
        st = L.lib().nvfp4_quantize_noalloc(x.data_ptr(), 0, n, None, 0, 0, 0, ts.data_ptr(),
                                            packed.data_ptr(), scales.data_ptr(), stream)
        assert st == 0

    call()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
