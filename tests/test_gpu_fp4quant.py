"""GPU parity: FP4Quant encode / decode for G in {64, 128, 256} through the
C ABI against the CPU oracle, bit for bit (codes, both scales, decoded
values)."""
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


def _check(x, G, out_dtype=torch.bfloat16):
    m = fp4()
    packed, s1, s2 = m.fp4quant_encode(x.to(dev()), G)
    xn = to_f32_np(x)
    wp, w1, w2 = ora.fp4quant_encode(xn, G)
    assert_bits_equal(to_f32_np(s1), w1, "s1")
    assert_bits_equal(to_f32_np(s2), w2, "s2")
    assert_bits_equal(u8(packed), wp, "packed")
    y = m.fp4quant_decode(packed, s1, s2, G, out_dtype)
    wy = ora.fp4quant_decode(wp, w1, w2, G)
    if out_dtype == torch.bfloat16:
        assert_bits_equal(bf16_bits(y), ora.bf16_rn(wy), "decoded bf16")
    else:
        assert_bits_equal(to_f32_np(y), wy, "decoded f32")


@pytest.mark.parametrize("G", [64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 256), (3, 512), (37, 4096), (1031, 768)])
def test_encode_decode_matches_oracle(G, dtype, rows, cols):
    x = workloads.fp4quant_acts(seed=rows, tokens=rows, hidden=cols, device="cpu").to(dtype)
    _check(x, G, torch.bfloat16 if dtype == torch.bfloat16 else torch.float32)


@pytest.mark.parametrize("G", [64, 128, 256])
def test_degenerate_groups(G):
    x = torch.zeros(4, 2 * G)
    x[0, 5] = 37.0                       # a single spike
    x[1, :] = 1.0                        # constant group
    x[2, G:] = -0.0
    x[3, :G] = torch.linspace(-1e-30, 1e-30, G)
    _check(x, G, torch.float32)


@pytest.mark.parametrize("G", [64, 128, 256])
def test_activation_workload_full_size_sampled(G):
    """bf16 [16384, 4096] Student-t(4) with 8 outlier channels x20: the whole
    tensor through the CUDA path, sampled rows against the oracle."""
    m = fp4()
    x = workloads.fp4quant_acts(seed=0, device=dev())
    packed, s1, s2 = m.fp4quant_encode(x, G)
    y = m.fp4quant_decode(packed, s1, s2, G)
    rng = np.random.default_rng(G)
    rows = torch.from_numpy(np.concatenate([[0, x.shape[0] - 1],
                                            rng.integers(0, x.shape[0], 40)])).to(dev())
    xs = to_f32_np(x[rows])
    wp, w1, w2 = ora.fp4quant_encode(xs, G)
    assert_bits_equal(to_f32_np(s1[rows]), w1, "s1")
    assert_bits_equal(to_f32_np(s2[rows]), w2, "s2")
    assert_bits_equal(u8(packed[rows]), wp, "packed")
    wy = ora.fp4quant_decode(wp, w1, w2, G)
    assert_bits_equal(bf16_bits(y[rows]), ora.bf16_rn(wy), "decoded")


@pytest.mark.parametrize("G", [64, 128, 256])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_groups_at_the_fp32_range_ends(G, out_dtype):
    """Groups whose sum of squares leaves the fp32 range: values near 2^64
    overflow it (RMS infinite, reciprocal 0, every transformed value 0, and
    the decode's 0 * infinity is NaN), values near 2^-64 underflow it (RMS
    0, the same zero path, decoding to zeros), and groups just inside both
    ends.  Codes and scales must match the oracle bit for bit; decoded
    values too, except that a NaN only has to be a NaN (its payload is not
    fixed)."""
    m = fp4()
    rng = np.random.default_rng(G)
    x = rng.standard_normal((6, 2 * G)).astype(np.float32)
    x[0, :G] *= np.float32(2.0 ** 64)          # squares overflow
    x[1, G:] *= np.float32(2.0 ** 60)          # inside
    x[2, :G] *= np.float32(2.0 ** -64)         # squares underflow to zero / subnormals
    x[3, G:] *= np.float32(2.0 ** -60)         # inside
    x[4, :G] = np.float32(3.0e38) * np.sign(x[4, :G])
    xt = torch.from_numpy(x)
    packed, s1, s2 = m.fp4quant_encode(xt.to(dev()), G)
    wp, w1, w2 = ora.fp4quant_encode(x, G)
    assert_bits_equal(to_f32_np(s1), w1, "s1")
    assert_bits_equal(to_f32_np(s2), w2, "s2")
    assert_bits_equal(u8(packed), wp, "packed")
    y = m.fp4quant_decode(packed, s1, s2, G, out_dtype)
    wy = ora.fp4quant_decode(wp, w1, w2, G)
    got = to_f32_np(y).astype(np.float32)
    nan = np.isnan(wy)
    assert np.array_equal(np.isnan(got), nan)
    if out_dtype == torch.bfloat16:
        assert_bits_equal(bf16_bits(y)[~nan], ora.bf16_rn(wy)[~nan], "decoded bf16")
    else:
        assert_bits_equal(got[~nan], wy[~nan], "decoded f32")


@pytest.mark.parametrize("G", [64, 128, 256])
@pytest.mark.parametrize("offset", [16, 1040])
def test_encode_input_inside_a_larger_buffer(G, offset):
    """The input as a view that starts `offset` bf16 elements (32 and 2080
    bytes) into a larger device buffer, with a ragged last tile: the G = 128
    bf16 encode reads it by TMA through a tensor map built on that address,
    the others by cp.async."""
    m = fp4()
    rows, cols = 45, 1024
    flat = workloads.fp4quant_acts(seed=offset, tokens=rows + 3, hidden=cols,
                                   device="cpu").to(torch.bfloat16).reshape(-1)
    d = flat.to(dev())
    x = d[offset:offset + rows * cols].view(rows, cols)
    assert x.data_ptr() % 32 == 0
    packed, s1, s2 = m.fp4quant_encode(x, G)
    wp, w1, w2 = ora.fp4quant_encode(to_f32_np(flat[offset:offset + rows * cols].view(rows, cols)), G)
    assert_bits_equal(to_f32_np(s1), w1, "s1")
    assert_bits_equal(to_f32_np(s2), w2, "s2")
    assert_bits_equal(u8(packed), wp, "packed")


def test_no_bounded_wait_gave_up():
    """No bounded wait in the library's kernels (the encode's TMA waits) gave
    up during the tests above."""
    assert fp4().wait_timeouts() == 0


@pytest.mark.timeout(120)
def test_bounded_wait_gives_up_and_the_context_survives():
    """The test hook announces the TMA copies of a one-tile bf16 G = 128
    encode 16 bytes longer than they are, so its one warp's wait never
    completes: the warp gives up after its limit, the timeout count grows by
    exactly one, and the next ordinary encode on the same context is exact."""
    from block_scaled_fp4_e2m1_gb300 import _lib
    m = fp4()
    x = workloads.fp4quant_acts(seed=5, tokens=2, hidden=256, device="cpu").to(torch.bfloat16)
    xd = x.to(dev())
    packed = torch.zeros(2 * 128, dtype=torch.uint8, device=dev())
    s1 = torch.zeros(4, dtype=torch.float32, device=dev())
    s2 = torch.zeros(4, dtype=torch.float32, device=dev())
    before = m.wait_timeouts()
    rc = _lib.lib().fp4_test_encode_wait_timeout(xd.data_ptr(), 2, 256, packed.data_ptr(),
                                                 s1.data_ptr(), s2.data_ptr(),
                                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert m.wait_timeouts() == before + 1
    _check(x, 128)
    assert m.wait_timeouts() == before + 1
