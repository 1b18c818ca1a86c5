"""GPU parity past 2^31 elements in a single tensor: NVFP4 amax, quantize
(RTN and SR) and dequantize, MXFP4 quantize and FP4Quant encode, on tensors
of just over 2^31 elements (4.3 GB of bf16 each), so that element and block
indices beyond the 32-bit range are exercised.  Sampled blocks and rows (the
first, those around element 2^31, random ones and the last) against the
oracle; the amax against an exact maximum."""
import numpy as np
import pytest
import torch

import oracle as ora
from parity_util import assert_bits_equal, bf16_bits, dev, ensure_built, to_f32_np, u8

pytestmark = pytest.mark.gpu

E31 = 2 ** 31


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def fp4():
    import block_scaled_fp4_e2m1_gb300 as m
    return m


def _gpu_bf16(n, seed, scale):
    g = torch.Generator(device=dev()).manual_seed(seed)
    return (torch.randn(n, generator=g, device=dev()) * scale).to(torch.bfloat16)


def _block_ranges(nb, rng, span=256):
    """Runs of `span` consecutive blocks: the first, around element 2^31,
    16 random ones and the last."""
    starts = [0, E31 // 16 - span // 2, nb - span] + list(rng.integers(0, nb - span, 16))
    return [(int(b0), span) for b0 in starts]


def test_nvfp4_single_tensor_past_2_31():
    m = fp4()
    n = E31 + 16 * 4096
    nb = n // 16
    x = _gpu_bf16(n, 123, 0.02)
    x[E31 + 5] = -0.9                                  # the amax sits past 2^31
    amax = m.nvfp4_amax(x)
    planted = abs(float(torch.tensor(-0.9).to(torch.bfloat16)))
    assert amax.item() == x.float().abs().max().item() == planted
    s_t = ora.nvfp4_tensor_scale(amax.item())
    rng = np.random.default_rng(1)
    for rounding in ("rtn", "sr"):
        packed, scales, ts = m.nvfp4_quantize(x, rounding=rounding, seed=9, step=3,
                                              tscale="compute")
        assert np.float32(ts.item()) == np.float32(s_t)
        y = m.nvfp4_dequantize(packed, scales, ts, (n,), torch.bfloat16)
        for b0, k in _block_ranges(nb, rng):
            v = to_f32_np(x[16 * b0:16 * (b0 + k)])
            wp, ws, _ = ora.nvfp4_blocks(v, b0, s_t, ora.SR if rounding == "sr" else ora.RTN,
                                         seed=9, step=3)
            assert_bits_equal(u8(packed[8 * b0:8 * (b0 + k)]), wp, f"packed {rounding} {b0}")
            assert_bits_equal(u8(scales[b0:b0 + k]), ws, f"scales {rounding} {b0}")
            wy = ora.nvfp4_dequantize(wp, ws, s_t, 16 * k)
            assert_bits_equal(bf16_bits(y[16 * b0:16 * (b0 + k)]), ora.bf16_rn(wy),
                              f"dequant {rounding} {b0}")
        del packed, scales, y


def test_mxfp4_quantize_past_2_31():
    m = fp4()
    cols = 7168
    rows = E31 // cols + 7
    x = _gpu_bf16(rows * cols, 7, 1.0).view(rows, cols)
    packed, scales = m.mxfp4_quantize(x)
    rng = np.random.default_rng(2)
    pick = sorted({0, E31 // cols - 1, E31 // cols, E31 // cols + 1, rows - 1}
                  | set(int(r) for r in rng.integers(0, rows, 12)))
    for r in pick:
        wp, ws = ora.mxfp4_quantize(to_f32_np(x[r:r + 1]))
        assert_bits_equal(u8(packed[r:r + 1]), wp, f"packed row {r}")
        assert_bits_equal(u8(scales[r:r + 1]), ws, f"scales row {r}")


def test_fp4quant_encode_past_2_31():
    m = fp4()
    cols, G = 4096, 128
    rows = E31 // cols + 16
    x = _gpu_bf16(rows * cols, 11, 1.0).view(rows, cols)
    packed, s1, s2 = m.fp4quant_encode(x, G)
    rng = np.random.default_rng(3)
    pick = sorted({0, E31 // cols - 1, E31 // cols, rows - 1}
                  | set(int(r) for r in rng.integers(0, rows, 12)))
    for r in pick:
        wp, w1, w2 = ora.fp4quant_encode(to_f32_np(x[r:r + 1]), G)
        assert_bits_equal(to_f32_np(s1[r:r + 1]), w1, f"s1 row {r}")
        assert_bits_equal(to_f32_np(s2[r:r + 1]), w2, f"s2 row {r}")
        assert_bits_equal(u8(packed[r:r + 1]), wp, f"packed row {r}")


def test_fp4_to_fp8_col_past_2_31_output_bytes():
    """The ragged column conversion with more than 2^31 output bytes: 64
    segments of random lengths over 299,600 dispatched rows x 7168.  The
    first and last segments, and the one holding output byte 2^31, against
    the per-segment oracle."""
    m = fp4()
    cols = 7168
    R = E31 // cols + 4000
    rng = np.random.default_rng(4)
    off = np.concatenate([[0], np.sort(rng.integers(0, R, 63)), [R]]).astype(np.int64)
    g = torch.Generator(device=dev()).manual_seed(5)
    pk = torch.randint(0, 256, (R, cols // 2), generator=g, device=dev(), dtype=torch.uint8)
    sc = torch.randint(110, 140, (R, cols // 32), generator=g, device=dev(), dtype=torch.uint8)
    segs = m.Segments(torch.from_numpy(off), dev())
    ft, fts = m.fp4_to_fp8_col(pk, sc, segs)
    sizes = np.diff(off)
    e_mid = int(np.searchsorted(off * cols, E31, side="right") - 1)
    assert off[e_mid] * cols <= E31 < off[e_mid + 1] * cols
    for e in sorted({0, e_mid, len(sizes) - 1}):
        row0, n_e = int(off[e]), int(sizes[e])
        if n_e == 0:
            continue
        wo, wsc = ora.fp4_to_fp8_col_segment(u8(pk[row0:row0 + n_e]), u8(sc[row0:row0 + n_e]),
                                             0, n_e)
        assert_bits_equal(u8(ft[cols * row0:cols * (row0 + n_e)]).reshape(cols, n_e), wo,
                          f"segment {e}")
        s0, nb = int(segs.scale_off_host[e]), (n_e + 127) // 128
        assert_bits_equal(to_f32_np(fts[cols * s0:cols * (s0 + nb)]).reshape(cols, nb), wsc,
                          f"segment {e} scales")
