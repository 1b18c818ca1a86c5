"""Pins for the oracle's FP4Quant encode / decode (CPU).

The FP4Quant page prints no numbers for the codec, so these pins are closed
forms and invariants: the normalized Walsh-Hadamard transform against
scipy's Sylvester Hadamard matrix (a library routine), unit vectors, exact
self-inverse on small integers, Parseval, the RMS scale against a float64
RMS, spike spreading, power-of-two invariance and the round-trip bound.
"""
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import oracle as ora

GROUPS = (64, 128, 256)


def test_wht_norm_constants():
    assert ora.wht_norm(64) == 0.125
    assert ora.wht_norm(256) == 0.0625
    c = np.float32(ora.wht_norm(128))
    assert c.view(np.uint32) == 0x3DB504F3
    # c is the float nearest to 2^-3.5: compare squares exactly
    below = np.nextafter(c, np.float32(0))
    above = np.nextafter(c, np.float32(1))
    target = Fraction(1, 128)
    sq = lambda f: Fraction(float(f)) ** 2
    assert (sq(below) < target < sq(above))
    mid_lo = (Fraction(float(below)) + Fraction(float(c))) / 2
    mid_hi = (Fraction(float(c)) + Fraction(float(above))) / 2
    assert mid_lo ** 2 < target < mid_hi ** 2


@pytest.mark.parametrize("G", GROUPS)
def test_wht_matches_sylvester_hadamard(G):
    rng = np.random.default_rng(G)
    H = scipy.linalg.hadamard(G).astype(np.float64) / np.sqrt(G)
    for _ in range(20):
        y = rng.standard_normal(G).astype(np.float32)
        got = ora.wht(y, G).astype(np.float64)
        want = H @ y.astype(np.float64)
        # log2(G) rounded butterfly stages + one scaling
        tol = (np.log2(G) + 2) * 2 ** -24 * np.sqrt(G) * np.abs(y).max()
        assert np.max(np.abs(got - want)) <= tol


@pytest.mark.parametrize("G", GROUPS)
def test_wht_unit_vectors(G):
    c = np.float32(ora.wht_norm(G))
    H = scipy.linalg.hadamard(G)
    for k in (0, 1, G // 2 - 1, G - 1):
        e = np.zeros(G, np.float32)
        e[k] = 1.0
        got = ora.wht(e, G)
        assert np.array_equal(got, (H[:, k] * c).astype(np.float32))


@pytest.mark.parametrize("G", (64, 256))
def test_wht_self_inverse_exact_on_integers(G):
    rng = np.random.default_rng(1)
    y = rng.integers(-50, 50, G).astype(np.float32)
    assert np.array_equal(ora.wht(ora.wht(y, G), G), y)
    const = np.ones(G, np.float32)
    z = ora.wht(const, G)
    assert z[0] == np.sqrt(G) and np.all(z[1:] == 0)


@pytest.mark.parametrize("G", GROUPS)
def test_wht_parseval_and_inverse(G):
    rng = np.random.default_rng(2)
    y = rng.standard_normal(G).astype(np.float32)
    z = ora.wht(y, G)
    assert abs(np.linalg.norm(z.astype(np.float64)) - np.linalg.norm(y.astype(np.float64))) \
        < 1e-5 * np.linalg.norm(y)
    back = ora.wht(z, G)
    assert np.max(np.abs(back - y)) < 1e-5 * np.abs(y).max() * np.log2(G)


@pytest.mark.parametrize("G", GROUPS)
def test_encode_scales(G):
    rng = np.random.default_rng(3)
    x = (rng.standard_t(4, (8, 4 * G))).astype(np.float32)
    packed, s1, s2 = ora.fp4quant_encode(x, G)
    xg = x.astype(np.float64).reshape(8, 4, G)
    rms = np.sqrt((xg ** 2).mean(-1))
    assert np.allclose(s1, rms, rtol=4e-7 * np.log2(G), atol=0)
    # after the RMS scale the group has unit RMS, so max|z| lies in [1, sqrt(G)]
    assert np.all(s2 >= 1.0 / 6 * (1 - 1e-6)) and np.all(s2 <= np.sqrt(G) / 6 * (1 + 1e-6))
    # s2 is max|WHT(x / s1)| / 6
    H = scipy.linalg.hadamard(G) / np.sqrt(G)
    z = (xg / s1[..., None].astype(np.float64)) @ H.T
    assert np.allclose(s2, np.abs(z).max(-1) / 6, rtol=1e-5)
    # the largest |z| in each group encodes to +-6
    codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(8, 4, G)
    assert np.all((codes & 7).max(-1) == 7)


@pytest.mark.parametrize("G", GROUPS)
def test_roundtrip_error_bound(G):
    rng = np.random.default_rng(4)
    x = (rng.standard_t(4, (16, 2 * G))).astype(np.float32)
    x[:, 3] *= 20
    packed, s1, s2 = ora.fp4quant_encode(x, G)
    y = ora.fp4quant_decode(packed, s1, s2, G)
    err = (y - x).astype(np.float64).reshape(16, 2, G)
    # per transformed coordinate the E2M1 error is at most one unit of s2
    # (half of the widest grid step, 2); the transform is orthogonal, so the
    # group error norm is at most s1 * s2 * sqrt(G) (plus fp32 noise)
    bound = s1.astype(np.float64) * s2 * np.sqrt(G) * (1 + 1e-3)
    assert np.all(np.linalg.norm(err, axis=-1) <= bound)


@pytest.mark.parametrize("G", GROUPS)
def test_spike_is_spread_and_recovered(G):
    """A single outlier is spread evenly by the transform: every coordinate
    becomes +-max and encodes to +-6, and decode gives the spike back."""
    x = np.zeros((1, G), np.float32)
    x[0, 5] = 37.0
    packed, s1, s2 = ora.fp4quant_encode(x, G)
    codes = np.stack([packed & 0xF, packed >> 4], -1).reshape(-1)
    assert np.all((codes & 7) == 7)
    y = ora.fp4quant_decode(packed, s1, s2, G)
    assert abs(y[0, 5] - 37.0) < 1e-4 and np.max(np.abs(np.delete(y[0], 5))) < 1e-4


@pytest.mark.parametrize("G", GROUPS)
def test_power_of_two_invariance_and_zero_group(G):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, G)).astype(np.float32)
    p1, a1, b1 = ora.fp4quant_encode(x, G)
    p2, a2, b2 = ora.fp4quant_encode(x * np.float32(8.0), G)
    assert np.array_equal(p1, p2) and np.array_equal(a2, a1 * 8) and np.array_equal(b1, b2)
    z = np.zeros((1, G), np.float32)
    p, a, b = ora.fp4quant_encode(z, G)
    assert np.all(p == 0) and a[0, 0] == 0 and b[0, 0] == 0
    assert np.all(ora.fp4quant_decode(p, a, b, G) == 0)


def test_bad_group_rejected():
    with pytest.raises(ValueError):
        ora.fp4quant_encode(np.zeros((1, 96), np.float32), 32)
    with pytest.raises(ValueError):
        ora.fp4quant_encode(np.zeros((1, 96), np.float32), 64)
