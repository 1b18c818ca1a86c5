"""GPU parity: one-scale-per-tensor E2M1 (the page's comparison point) and
the four round trips of the quality report against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle as ora
from block_scaled_fp4_e2m1_gb300 import workloads
from parity_util import assert_bits_equal, bf16_bits, dev, ensure_built, to_f32_np, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def fp4():
    import block_scaled_fp4_e2m1_gb300 as m
    return m


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("scale", [1.0, 0.2016666, 3.7e-5, 2.0 ** -20, 1e30])
def test_scaled_round_trip_matches_oracle(dtype, scale):
    m = fp4()
    g = torch.Generator().manual_seed(11)
    n = 16 * 4099
    x = (torch.randn(n, generator=g) * torch.exp2(torch.randint(-30, 30, (n,), generator=g).float()))
    x = x.clamp(-3e38, 3e38).to(dtype)
    pk = m.fp4_scaled_quantize(x.to(dev()), scale)
    wp = ora.fp4_scaled_quantize(to_f32_np(x), scale)
    assert_bits_equal(u8(pk), wp, "packed")
    for od in (torch.float32, torch.bfloat16):
        y = m.fp4_scaled_dequantize(pk, n, scale, od)
        wy = ora.fp4_scaled_dequantize(wp, n, scale)
        if od == torch.bfloat16:
            assert_bits_equal(bf16_bits(y), ora.bf16_rn(wy), "y bf16")
        else:
            assert_bits_equal(to_f32_np(y), wy, "y f32")


def test_quality_report_round_trips_and_stats():
    """One synthetic down_proj-shaped matrix (Laplace weights with outliers):
    the four stored tensors equal the oracle's, and the statistics follow
    from them."""
    m = fp4()
    from block_scaled_fp4_e2m1_gb300 import quality
    w = workloads.laplace_weight(18, (512, 1536), device=dev())
    rt = quality.round_trips(w)
    wn = to_f32_np(w).reshape(-1)
    amax = np.float32(np.abs(wn).max())
    s = np.float32(amax / np.float32(6.0))
    want = {
        "straight": ora.fp4_scaled_dequantize(ora.fp4_scaled_quantize(wn, 1.0), wn.size, 1.0),
        "per_matrix": ora.fp4_scaled_dequantize(ora.fp4_scaled_quantize(wn, s), wn.size, s),
        "mxfp4": ora.mxfp4_dequantize(*ora.mxfp4_quantize(wn.reshape(512, 1536))).reshape(-1),
    }
    pk, sc, ts = ora.nvfp4_quantize(wn)
    want["nvfp4"] = ora.nvfp4_dequantize(pk, sc, ts, wn.size)
    rep = m.fp4_quality(w)
    for k, q in want.items():
        assert_bits_equal(to_f32_np(rt[k]).reshape(-1), q, k)
        zero = int(np.count_nonzero(q == 0)) / q.size
        err = float(np.abs(wn.astype(np.float64) - q).sum() / np.abs(wn.astype(np.float64)).sum())
        assert rep[k]["zero"] == zero
        assert rep[k]["error"] == pytest.approx(err, rel=1e-12)
    # the page's ordering: block scaling far ahead, NVFP4 ahead of MXFP4
    assert rep["straight"]["zero"] > 0.99 and rep["per_matrix"]["zero"] > 0.5
    assert rep["nvfp4"]["error"] < rep["mxfp4"]["error"] < rep["per_matrix"]["error"]


def test_scale_from_amax_on_the_device():
    """fp4_scaled_quantize_amax forms RN(amax / 6) on the device: codes and
    the published scale equal the oracle's with that scale; an all-zero
    tensor (amax 0) and an empty one publish scale 1."""
    m = fp4()
    x = workloads.laplace_weight(21, (64, 256), device=dev()).view(-1)
    xn = to_f32_np(x)
    amax = m.nvfp4_amax(x)
    pk, s = m.fp4_scaled_quantize_amax(x, amax)
    want_s = np.float32(np.float32(np.abs(xn).max()) / np.float32(6.0))
    assert np.float32(s.item()) == want_s
    assert_bits_equal(u8(pk), ora.fp4_scaled_quantize(xn, float(want_s)), "codes")
    for od in (torch.float32, torch.bfloat16):
        y = m.fp4_scaled_dequantize_dev(pk, x.numel(), s, od)
        wy = ora.fp4_scaled_dequantize(u8(pk), x.numel(), float(want_s))
        got = to_f32_np(y) if od == torch.float32 else bf16_bits(y)
        assert_bits_equal(got, wy if od == torch.float32 else ora.bf16_rn(wy), str(od))
    zero = torch.zeros(256, dtype=torch.bfloat16, device=dev())
    _, s0 = m.fp4_scaled_quantize_amax(zero, m.nvfp4_amax(zero))
    assert s0.item() == 1.0
    empty = torch.empty(0, dtype=torch.float32, device=dev())
    s1 = torch.full((1,), -3.0, device=dev())
    m.fp4_scaled_quantize_amax(empty, torch.zeros(1, device=dev()), scale_out=s1)
    assert s1.item() == 1.0
