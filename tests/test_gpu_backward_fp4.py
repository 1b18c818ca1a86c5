"""GPU parity: the backward-path FP4 calls (FP8 -> MXFP4 quantize, MXFP4
dequantize) through the C ABI against the CPU oracle, bit for bit."""
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


def _fp8_grads(rows, cols, seed):
    """E4M3 bytes of every finite value (no NaN bytes), with fp32 block
    scales spanning many binades (powers of two and arbitrary values)."""
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 256, (rows, cols)).astype(np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x3C
    s = (rng.uniform(0.5, 2.0, (rows, cols // 128)) * np.exp2(rng.integers(-60, 60, (rows, cols // 128)))).astype(np.float32)
    s[:, ::3] = np.exp2(rng.integers(-30, 30, s[:, ::3].shape)).astype(np.float32)
    return b, s


@pytest.mark.parametrize("rows,cols", [(1, 128), (7, 384), (129, 7168), (1000, 256)])
def test_fp8_to_fp4_row_matches_oracle(rows, cols):
    m = fp4()
    b, s = _fp8_grads(rows, cols, seed=rows)
    pk, sc = m.fp8_to_fp4_row(torch.from_numpy(b).to(dev()), torch.from_numpy(s).to(dev()))
    wp, ws = ora.fp8_to_fp4_row(b, s)
    assert_bits_equal(u8(sc), ws, "scales")
    assert_bits_equal(u8(pk), wp, "packed")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (257, 7168)])
def test_mxfp4_dequantize_matches_oracle(out_dtype, rows, cols):
    m = fp4()
    rng = np.random.default_rng(cols + rows)
    pk = rng.integers(0, 256, (rows, cols // 2)).astype(np.uint8)
    sc = rng.integers(0, 256, (rows, cols // 32)).astype(np.uint8)   # every byte, 255 included
    sc.reshape(-1)[:256] = np.arange(256, dtype=np.uint8)[: sc.size]
    y = m.mxfp4_dequantize(torch.from_numpy(pk).to(dev()), torch.from_numpy(sc).to(dev()), out_dtype)
    wy = ora.mxfp4_dequantize(pk, sc)
    if out_dtype == torch.bfloat16:
        assert_bits_equal(bf16_bits(y), ora.bf16_rn(wy), "y bf16")
    else:
        assert_bits_equal(to_f32_np(y), wy, "y f32")


def test_backward_exchange_on_moe_shapes():
    """A gradient block of the MoE shape through the whole exchange: bf16 ->
    MXFP4 -> FP8 (FP4RowToFP8Row) -> MXFP4 (this call) -> bf16, every stage
    against the oracle."""
    m = fp4()
    x = workloads.moe_tokens(seed=3, tokens=64, hidden=7168, device=dev())
    pk, sc = m.mxfp4_quantize(x)
    f8, fs = m.fp4_to_fp8_row(pk, sc)
    p2, s2 = m.fp8_to_fp4_row(f8, fs)
    y = m.mxfp4_dequantize(p2, s2, torch.bfloat16)
    wpk, wsc = ora.mxfp4_quantize(to_f32_np(x))
    wf8, wfs = ora.fp4_to_fp8_row(wpk, wsc)
    wp2, ws2 = ora.fp8_to_fp4_row(wf8, wfs)
    assert_bits_equal(u8(f8), wf8, "fp8")
    assert_bits_equal(u8(p2), wp2, "packed")
    assert_bits_equal(u8(s2), ws2, "scales")
    assert_bits_equal(bf16_bits(y), ora.bf16_rn(ora.mxfp4_dequantize(wp2, ws2)), "y")


def test_fp8_to_fp4_row_extreme_scales():
    """FP8 -> MXFP4 where the products leave the normal range: per-128 scales
    from the smallest subnormal up to the largest float, so that
    e4m3 * scale underflows to subnormals or zero, or overflows to infinity
    (which the MXFP4 rule saturates to +-6 under its largest exponent); also
    all-zero blocks, blocks of -0 bytes and single-value blocks."""
    m = fp4()
    rows, cols = 48, 512
    rng = np.random.default_rng(77)
    b = rng.integers(0, 256, (rows, cols)).astype(np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x3C                       # no NaN bytes
    b[0, :32] = 0
    b[1, :32] = 0x80                                    # -0
    b[2, :32] = 0
    b[2, 5] = 0x7E                                      # 448 alone
    b[3, 32:64] = 0xFE                                  # -448 everywhere
    ext = np.array([2.0 ** -149, 2.0 ** -140, 2.0 ** -126, 1e-30, 1.0, 2.0 ** 60, 2.0 ** 100,
                    2.0 ** 120, 2.0 ** 126, 2.0 ** 127, 3.4e38, 0.75 * 2.0 ** -133],
                   dtype=np.float32)
    s = ext[rng.integers(0, ext.size, (rows, cols // 128))]
    pk, sc = m.fp8_to_fp4_row(torch.from_numpy(b).to(dev()), torch.from_numpy(s).to(dev()))
    wp, ws = ora.fp8_to_fp4_row(b, s)
    assert_bits_equal(u8(sc), ws, "scales")
    assert_bits_equal(u8(pk), wp, "packed")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mxfp4_quantize_infinite_inputs(dtype):
    """mxfp4_quantize on blocks holding +-infinity beside finite values and
    beside blocks without one: the same rule as the oracle (exponent from
    the amax's exponent field, infinities saturated to +-6)."""
    m = fp4()
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 256)).astype(np.float32)
    x[0, 3] = np.inf
    x[1, 40] = -np.inf
    x[2, :32] = np.inf
    x[3, 100] = np.inf
    x[3, 101] = -np.inf
    xt = torch.from_numpy(x).to(dtype)
    pk, sc = m.mxfp4_quantize(xt.to(dev()))
    wp, ws = ora.mxfp4_quantize(to_f32_np(xt))
    assert_bits_equal(u8(sc), ws, "scales")
    assert_bits_equal(u8(pk), wp, "packed")
