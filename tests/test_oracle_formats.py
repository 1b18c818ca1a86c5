"""Pins for the oracle's format helpers (CPU only).

E2M1: the page's table, its worked thresholds, and a second, independent
formulation of round-to-nearest-even (scaling by the binade's quantum).
E4M3 and bf16: PyTorch's own CPU conversions (library routines).
"""
import math

import numpy as np
import pytest
import torch

import oracle as ora
from golden_util import load

E2M1_VALUES = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def test_e2m1_table_matches_page():
    g = load("e2m1_grid.txt")
    rows = g["_rows"]
    assert len(rows) == 8
    for ebits, mbit, value in rows:
        code = (int(ebits, 2) << 1) | int(mbit)
        assert ora.e2m1_value([code])[0] == float(value)
        # the sign bit gives the negative copy
        assert ora.e2m1_value([code | 8])[0] == -float(value) or float(value) == 0.0
        assert math.copysign(1.0, ora.e2m1_value([code | 8])[0]) == -1.0


def _e2m1_by_quantum(a: float) -> int:
    """RNE to a 1-mantissa-bit format with exponent bias 1: scale by the
    quantum of the binade, round half to even (Python round), saturate."""
    sign = 8 if math.copysign(1.0, a) < 0 else 0
    m = abs(a)
    if m >= 6.0:
        return sign | 7
    e = 0 if m == 0 else max(math.floor(math.log2(m)), 0)
    q = 2.0 ** (e - 1)
    val = round(m / q) * q
    if val > 6.0:
        val = 6.0
    return sign | E2M1_VALUES[val]


def _sample_floats(rng):
    bf16 = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    bf16 = bf16[np.isfinite(bf16)]
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 6.0, 0.0], np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)),
                           np.nextafter(mids, np.float32(-np.inf))])
    near = np.concatenate([near, -near])
    rnd = rng.uniform(-9, 9, 20000).astype(np.float32)
    tiny = (rng.standard_normal(2000) * 1e-30).astype(np.float32)
    return np.concatenate([bf16, near, rnd, tiny])


def test_e2m1_rn_matches_quantum_rounding():
    rng = np.random.default_rng(1)
    xs = _sample_floats(rng)
    got = ora.e2m1_rn(xs)
    want = np.array([_e2m1_by_quantum(float(x)) for x in xs], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], got[i], want[i]) for i in bad[:10]]


def test_e2m1_rn_page_thresholds():
    w = load("worked_block.txt")
    thr = float(w["zero_threshold"][0])
    # below 0.25 -> 0; 0.25 is the midpoint and ties to the even code 0
    assert ora.e2m1_rn([np.nextafter(np.float32(thr), np.float32(0))])[0] == 0
    assert ora.e2m1_rn([thr])[0] == 0
    assert ora.e2m1_rn([np.nextafter(np.float32(thr), np.float32(1))])[0] == 1
    # the page's four weights rounded straight to FP4 are all 0 (sign kept)
    codes = ora.e2m1_rn([float(v) for v in w["weights"]])
    assert all(ora.e2m1_value(codes) == 0.0)
    # ties to even mantissa: 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    got = ora.e2m1_value(ora.e2m1_rn([0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -7.0]))
    assert list(got) == [1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -6.0]


def test_e4m3_decode_all_codes():
    vals = ora.e4m3_value(np.arange(256))
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    fin = ~np.isnan(t)
    assert np.array_equal(np.isnan(vals), np.isnan(t))
    assert np.array_equal(vals[fin], t[fin].astype(np.float64))
    assert ora.e4m3_value([0x7E])[0] == 448.0
    assert ora.e4m3_value([0x01])[0] == 2.0 ** -9


def test_e4m3_rn_matches_torch():
    rng = np.random.default_rng(2)
    bf16 = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    xs = np.concatenate([bf16, rng.standard_normal(50000).astype(np.float32) * 3,
                         rng.uniform(0, 2 ** -6, 20000).astype(np.float32),
                         ora.e4m3_value(np.arange(0, 126)).astype(np.float32)])
    xs = xs[np.isfinite(xs) & (np.abs(xs) < 464.0)]
    # midpoints between adjacent e4m3 values (exact in fp32): ties to even
    pos = ora.e4m3_value(np.arange(0, 127))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    xs = np.concatenate([xs, mids, -mids])
    got = ora.e4m3_rn(xs.astype(np.float64))
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], got[i], want[i]) for i in bad[:10]]


def test_e4m3_saturates():
    assert list(ora.e4m3_rn([464.0, 500.0, 1e30, -1e9])) == [0x7E, 0x7E, 0x7E, 0xFE]


def test_bf16_rn_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2 ** 16, 5000, dtype=np.uint32) << 16) | 0x8000
    xs = np.concatenate([bits, ties]).view(np.float32)
    xs = xs[np.isfinite(xs)]
    got = ora.bf16_rn(xs)
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_ue8m0_values():
    v = ora.ue8m0_value(np.arange(255))
    assert np.array_equal(v, 2.0 ** (np.arange(255) - 127.0))
