"""Pins for the oracle's blocked (swizzled) block-scale layout (CPU).

The pages only name the layout ([fp4-train] "Scope": scales swizzled into the
layout torch._scaled_mm consumes).  The oracle is pinned here against
PyTorch's own helper that prepares block scales for torch._scaled_mm (an
independent implementation of the same layout, shipped with PyTorch's test
utilities), and by invariants: a bijection of the padded index space, zero
padding, and an exact inverse.  The GPU test ``test_gpu_blocked_scales.py``
adds the consumer itself: torch._scaled_mm on scales laid out by the oracle.
"""
import ast
import os

import numpy as np
import pytest
import torch

import oracle as ora

SHAPES = [(1, 1), (128, 4), (129, 5), (256, 8), (300, 22), (5, 257), (1000, 3), (384, 64)]


def _torch_blocked_helper():
    """torch's to_blocked (and the ceil_div it uses), taken from the source
    of torch/testing/_internal/common_quantized.py without importing that
    module (its imports need test-only packages)."""
    path = os.path.join(os.path.dirname(torch.__file__), "testing", "_internal",
                        "common_quantized.py")
    if not os.path.exists(path):
        pytest.skip("torch's quantized test helpers are not installed")
    tree = ast.parse(open(path).read())
    wanted = {"ceil_div", "to_blocked"}
    fns = [n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name in wanted]
    if {f.name for f in fns} != wanted:
        pytest.skip("torch's to_blocked helper is not in this PyTorch version")
    ns = {"torch": torch, "Tensor": torch.Tensor}
    exec(compile(ast.Module(body=fns, type_ignores=[]), path, "exec"), ns)
    return ns["to_blocked"]


def _labels(rows, cols):
    """Distinct non-zero 24-bit labels 1 .. rows*cols in row-major order."""
    return np.arange(1, rows * cols + 1, dtype=np.uint32).reshape(rows, cols)


def _blocked_labels(lab, rows, cols):
    """Push each byte plane of the labels through the oracle and rejoin."""
    out = np.zeros(ora.blocked_scales_size(rows, cols), dtype=np.uint32)
    for k in range(3):
        plane = ((lab >> (8 * k)) & 0xFF).astype(np.uint8)
        out |= ora.scales_to_blocked(plane, rows, cols).astype(np.uint32) << (8 * k)
    return out


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_matches_pytorch_scaled_mm_helper(rows, cols):
    to_blocked = _torch_blocked_helper()
    rng = np.random.default_rng(rows * 1000 + cols)
    s = rng.integers(1, 256, (rows, cols), dtype=np.uint8)
    want = to_blocked(torch.from_numpy(s)).reshape(-1).numpy()
    got = ora.scales_to_blocked(s, rows, cols)
    assert got.size == want.size
    assert np.array_equal(got, want)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_size_is_whole_tiles(rows, cols):
    prow = -(-rows // 128) * 128
    pcol = -(-cols // 4) * 4
    assert ora.blocked_scales_size(rows, cols) == prow * pcol
    assert ora.blocked_scales_size(rows, cols) % 512 == 0


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_bijection_padding_and_inverse(rows, cols):
    lab = _labels(rows, cols)
    b = _blocked_labels(lab, rows, cols)
    # every scale appears exactly once, every other byte is padding (0)
    nz = b[b != 0]
    assert nz.size == rows * cols
    assert np.array_equal(np.sort(nz), lab.reshape(-1))
    # the inverse reads every scale back
    rng = np.random.default_rng(7)
    s = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
    assert np.array_equal(ora.scales_from_blocked(ora.scales_to_blocked(s, rows, cols),
                                                  rows, cols), s)


def test_tile_geometry():
    """Within one 512-byte tile, each 16-byte line holds rows i, i+32, i+64
    and i+96 with their four consecutive scales; tiles follow row-major order
    over [row tile, column tile]."""
    rows, cols = 256, 8
    lab = _labels(rows, cols)
    b = _blocked_labels(lab, rows, cols).reshape(2, 2, 32, 4, 4)   # [rt, ct, i, g, c]
    for rt in range(2):
        for ct in range(2):
            for i in range(32):
                for g in range(4):
                    r = 128 * rt + 32 * g + i
                    assert list(b[rt, ct, i, g]) == list(lab[r, 4 * ct:4 * ct + 4])


def test_negative_sizes_rejected():
    assert ora.blocked_scales_size(-1, 4) == -1
    assert ora.lib().ora_scales_to_blocked(None, -1, 4, None) == 1
    assert ora.lib().ora_scales_from_blocked(None, 4, -1, None) == 1
