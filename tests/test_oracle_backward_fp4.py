"""Pins for the oracle's backward-path FP4 operations (CPU): MXFP4
dequantize, and FP8 (E4M3 with per-128 fp32 scales) -> MXFP4 quantize.

[MoE-FP4] "方法概述" keeps gradients in FP8 and "局限与未来方向" names FP4 for
the backward pass as future work: gradients in FP8 become MXFP4 for the
exchange and come back to FP8 (FP4RowToFP8Row) or to floats (dequantize).
"""
from fractions import Fraction

import numpy as np

import oracle as ora
from golden_util import load


def _grid():
    """E2M1 code -> exact value from the page's table (codes 8..15 negative)."""
    rows = load("e2m1_grid.txt")["_rows"]
    pos = [Fraction(r[2]) for r in rows]
    return pos + [-v for v in pos]


def test_mxfp4_dequantize_is_the_exact_product():
    """Every code under every UE8M0 byte that keeps the product in the normal
    fp32 range: value(code) * 2^(S - 127) exactly (Fraction arithmetic from
    the page's table)."""
    grid = _grid()
    S = np.arange(3, 252, dtype=np.uint8)           # 2^-124 .. 2^124
    codes = np.arange(16, dtype=np.uint8)
    packed = np.zeros((S.size, 16), np.uint8)        # 32 codes per row: 0..15, 0..15
    packed[:, :8] = (codes[0::2] | (codes[1::2] << 4))
    packed[:, 8:] = packed[:, :8]
    scales = S.reshape(-1, 1)
    y = ora.mxfp4_dequantize(packed, scales)
    for r, s in enumerate(S):
        want = [float(grid[c] * Fraction(2) ** (int(s) - 127)) for c in range(16)] * 2
        assert y[r].tolist() == [float(np.float32(w)) for w in want], s


def test_mxfp4_quantize_dequantize_identity_on_the_grid():
    """Values already on an MXFP4 grid whose block maximum has magnitude 4 or
    6 quantize back to the same codes and scale."""
    rng = np.random.default_rng(3)
    grid = np.array([float(v) for v in _grid()], np.float64)
    for E in (-120, -30, -3, 0, 7, 60, 120):
        c = rng.integers(0, 16, (8, 32))
        c[:, 0] = rng.choice([6, 7, 14, 15], 8)       # +-4 or +-6 in every block
        x = (grid[c] * 2.0 ** E).astype(np.float32)
        packed, scales = ora.mxfp4_quantize(x)
        assert np.all(scales == E + 127)
        assert np.array_equal(ora.mxfp4_dequantize(packed, scales), x)


def test_fp8_round_trip_preserves_values():
    """MXFP4 -> FP8 (FP4RowToFP8Row) -> MXFP4 returns the same values while
    the FP8 step is exact (block scales within 8 of their 128-block's
    largest), even where the codes and scales are not the same."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 512)) * np.exp2(rng.integers(-4, 5, (16, 512)))).astype(np.float32)
    packed, scales = ora.mxfp4_quantize(x)
    s4 = scales.reshape(16, -1, 4)
    assert np.all(s4.max(-1, keepdims=True) - s4 <= 8)
    fp8, fsc = ora.fp4_to_fp8_row(packed, scales)
    p2, s2 = ora.fp8_to_fp4_row(fp8, fsc)
    assert np.array_equal(ora.mxfp4_dequantize(p2, s2), ora.mxfp4_dequantize(packed, scales))


def test_fp8_to_fp4_under_unit_scale_is_mxfp4_of_the_e4m3_values():
    """With every fp32 block scale 1 the operation reduces to MXFP4 quantize
    of the decoded E4M3 values (all 254 finite bytes appear)."""
    rng = np.random.default_rng(5)
    b = rng.integers(0, 256, (32, 256)).astype(np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x00                      # no NaN bytes
    b[0, :254] = [v for v in range(256) if (v & 0x7F) != 0x7F]
    ones = np.ones((32, 2), np.float32)
    p, s = ora.fp8_to_fp4_row(b, ones)
    pw, sw = ora.mxfp4_quantize(ora.e4m3_value(b).astype(np.float32))
    assert np.array_equal(p, pw) and np.array_equal(s, sw)


def test_fp8_to_fp4_power_of_two_scale_shifts_only_the_exponent():
    """Multiplying a block's fp32 scale by 2^k leaves the codes unchanged and
    adds k to the UE8M0 bytes (in range)."""
    rng = np.random.default_rng(6)
    b = rng.integers(0, 0x7E, (8, 256)).astype(np.uint8) | (rng.integers(0, 2, (8, 256)) << 7).astype(np.uint8)
    base = np.full((8, 2), 0.5, np.float32)
    p0, s0 = ora.fp8_to_fp4_row(b, base)
    for k in (-20, -1, 3, 17):
        pk, sk = ora.fp8_to_fp4_row(b, (base * np.float32(2.0 ** k)).astype(np.float32))
        assert np.array_equal(pk, p0)
        assert np.array_equal(sk.astype(int), s0.astype(int) + k)
