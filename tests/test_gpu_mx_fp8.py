"""GPU parity: MXFP4 quantize, FP4 -> FP8 row and ragged column conversion,
against the CPU oracle, bit for bit; plus exhaustive checks of the device's
E2M1 and E4M3 rounding (through the public kernels) against the oracle's."""
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


def _e2m1_probe(values: np.ndarray) -> np.ndarray:
    """E2M1 codes the device gives |values| < 8, read through mxfp4_quantize:
    each 32-block holds 31 test values and an anchor 4.0, so its exponent is
    0 and the codes are RN_e2m1(value) itself."""
    m = fp4()
    n = values.size
    nb = (n + 30) // 31
    blk = np.zeros((nb, 32), np.float32)
    flat = np.zeros(nb * 31, np.float32)
    flat[:n] = values
    blk[:, :31] = flat.reshape(nb, 31)
    blk[:, 31] = 4.0
    x = torch.from_numpy(blk).to(dev())
    packed, scales = m.mxfp4_quantize(x)
    assert np.all(u8(scales) == 127)
    p = u8(packed).reshape(nb, 16)
    codes = np.stack([p & 0xF, p >> 4], axis=-1).reshape(nb, 32)[:, :31].ravel()[:n]
    return codes


def test_e2m1_rounding_exhaustive_in_rounding_range():
    """Every fp32 with 2^-3 <= |x| < 8 (all 2^23 mantissas of 6 binades, both
    signs), plus every finite bf16 below 8, plus zeros and subnormals."""
    exps = np.arange(124, 130, dtype=np.uint32)
    mant = np.arange(1 << 23, dtype=np.uint32)
    for e in exps:
        for sign in (0, 1):
            bits = (np.uint32(sign) << 31) | (e << 23) | mant
            vals = bits.view(np.float32)
            got = _e2m1_probe(vals)
            want = ora.e2m1_rn(vals)
            assert_bits_equal(got, want, f"e2m1 exp {e} sign {sign}")
    bf = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf) & (np.abs(bf) < 8)]
    extra = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-38, -1e-38], np.float32)
    vals = np.concatenate([bf, extra])
    assert_bits_equal(_e2m1_probe(vals), ora.e2m1_rn(vals), "e2m1 bf16 + specials")


def _e4m3_probe(values: np.ndarray) -> np.ndarray:
    """E4M3 scale bytes the device gives non-negative values through
    nvfp4_quantize: each block holds one value; with a given tensor scale
    1/6 the block scale is RN_e4m3(value)."""
    m = fp4()
    n = values.size
    x = np.zeros((n, 16), np.float32)
    x[:, 5] = values
    ts = torch.full((1,), float(np.float32(1.0) / np.float32(6.0)), dtype=torch.float32,
                    device=dev())
    assert np.float32(6.0) * np.float32(ts.item()) == np.float32(1.0)
    _, scales, _ = m.nvfp4_quantize(torch.from_numpy(x.ravel()).to(dev()), tscale="given",
                                    tensor_scale=ts)
    return u8(scales)


def test_e4m3_rounding():
    rng = np.random.default_rng(0)
    pos = ora.e4m3_value(np.arange(0, 127))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1e9)), pos.astype(np.float32)])
    bf = (np.arange(0, 1 << 15, dtype=np.uint32) << 16).view(np.float32)
    bf = bf[np.isfinite(bf)]
    dense = (np.uint32(rng.integers(0x3A000000, 0x43F00000, 1 << 22, dtype=np.int64))
             .astype(np.uint32).view(np.float32))
    vals = np.concatenate([near, bf, dense, np.array([448.0, 464.0, 500.0, 3e38], np.float32)])
    got = _e4m3_probe(vals)
    want = ora.e4m3_rn(vals.astype(np.float64))
    assert_bits_equal(got, want, "e4m3")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (257, 7168), (1000, 224)])
def test_mxfp4_quantize_matches_oracle(dtype, rows, cols):
    m = fp4()
    g = torch.Generator().manual_seed(rows * cols)
    x = (torch.randn(rows, cols, generator=g) * torch.exp(torch.randn(rows, 1, generator=g) * 4))
    x = x.to(dtype)
    packed, scales = m.mxfp4_quantize(x.to(dev()))
    wp, ws = ora.mxfp4_quantize(to_f32_np(x))
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")


def test_mxfp4_degenerate_blocks():
    m = fp4()
    x = np.zeros((2, 128), np.float32)
    x[0, 32:64] = -0.0
    x[0, 64] = 1e-42
    x[0, 96:128] = np.float32(3.3e38)
    x[1, :32] = np.float32(7.999)
    x[1, 32:64] = np.float32(2.0 ** -130)
    x[1, 64:96] = np.linspace(-8, 8, 32, dtype=np.float32)
    packed, scales = m.mxfp4_quantize(torch.from_numpy(x).to(dev()))
    wp, ws = ora.mxfp4_quantize(x)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")


def test_fp4_to_fp8_row_all_codes_all_shifts():
    """All 16 codes under every shift S_t - S_sub in [0, 254]."""
    m = fp4()
    rows = 255
    packed = np.zeros((rows, 64), np.uint8)
    codes = np.tile(np.arange(16, dtype=np.uint8), 8)
    packed[:] = codes[0::2] | (codes[1::2] << 4)
    scales = np.zeros((rows, 4), np.uint8)
    for d in range(rows):
        scales[d] = [254, 254 - d, (254 - d // 2), 127] if d <= 127 else [254, 254 - d, 200, 0]
    fp8, fsc = m.fp4_to_fp8_row(torch.from_numpy(packed).to(dev()),
                                torch.from_numpy(scales).to(dev()))
    wf, wfs = ora.fp4_to_fp8_row(packed, scales)
    assert_bits_equal(u8(fp8), wf, "fp8")
    assert_bits_equal(to_f32_np(fsc), wfs, "scales")


@pytest.mark.parametrize("rows,cols", [(1, 128), (7, 256), (300, 7168), (4099, 384)])
def test_fp4_to_fp8_row_matches_oracle(rows, cols):
    m = fp4()
    rng = np.random.default_rng(rows)
    packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (rows, cols // 32), dtype=np.uint8)
    scales[0, 0] = 0
    fp8, fsc = m.fp4_to_fp8_row(torch.from_numpy(packed).to(dev()),
                                torch.from_numpy(scales).to(dev()))
    wf, wfs = ora.fp4_to_fp8_row(packed, scales)
    assert_bits_equal(u8(fp8), wf, "fp8")
    assert_bits_equal(to_f32_np(fsc), wfs, "scales")


SEGMENT_SETS = [
    [5],
    [128],
    [129, 0, 1, 127, 128, 0],
    [0, 0, 0, 300],
    [1, 2, 3, 250, 513, 77, 131, 0, 64],
    list(range(1, 50)),                   # every row start / end alignment
    [17 * k + 3 for k in range(12)],
]


@pytest.mark.parametrize("sizes", SEGMENT_SETS)
@pytest.mark.parametrize("cols", [128, 384])
def test_fp4_to_fp8_col_ragged_matches_oracle(sizes, cols):
    m = fp4()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    rng = np.random.default_rng(R + cols)
    packed = rng.integers(0, 256, (max(R, 1), cols // 2), dtype=np.uint8)[:R]
    scales = rng.integers(115, 135, (max(R, 1), cols // 32), dtype=np.uint8)[:R]
    segs = m.Segments(torch.from_numpy(off), dev())
    pk = torch.from_numpy(np.ascontiguousarray(packed)).to(dev())
    sc = torch.from_numpy(np.ascontiguousarray(scales)).to(dev())
    # canary around the outputs
    out = torch.full((cols * R + 64,), 0xA5, dtype=torch.uint8, device=dev())
    osc = torch.full((cols * segs.total_blocks + 16,), -7.0, dtype=torch.float32, device=dev())
    m.fp4_to_fp8_col(pk, sc, segs, out[32:32 + cols * R], osc[8:8 + cols * segs.total_blocks])
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    o = u8(out)
    assert np.all(o[:32] == 0xA5) and np.all(o[32 + cols * R:] == 0xA5)
    assert_bits_equal(o[32:32 + cols * R], wo, "fp8_t")
    s = to_f32_np(osc)
    assert np.all(s[:8] == -7.0) and np.all(s[8 + cols * segs.total_blocks:] == -7.0)
    assert_bits_equal(s[8:8 + cols * segs.total_blocks], wsc, "fp8_t scales")


def test_moe_workload_reduced_end_to_end():
    """The MoE path at reduced size: bf16 tokens -> MXFP4 rows, dispatch
    gather (top-8 of 256 Zipf experts), row and column FP8 conversion."""
    m = fp4()
    T, H, E = 512, 7168, 256
    x = workloads.moe_tokens(seed=0, tokens=T, hidden=H, device=dev())
    row_token, row_off = workloads.moe_routing(seed=0, tokens=T, experts=E)
    packed, scales = m.mxfp4_quantize(x)
    xn = to_f32_np(x)
    wp, ws = ora.mxfp4_quantize(xn)
    assert_bits_equal(u8(packed), wp, "mxfp4 packed")
    assert_bits_equal(u8(scales), ws, "mxfp4 scales")
    idx = row_token.to(dev())
    dp = packed.index_select(0, idx).contiguous()
    ds = scales.index_select(0, idx).contiguous()
    fp8, fsc = m.fp4_to_fp8_row(dp, ds)
    wf, wfs = ora.fp4_to_fp8_row(wp[row_token.numpy()], ws[row_token.numpy()])
    assert_bits_equal(u8(fp8), wf, "row fp8")
    assert_bits_equal(to_f32_np(fsc), wfs, "row scales")
    segs = m.Segments(row_off, dev())
    ft, fts = m.fp4_to_fp8_col(dp, ds, segs)
    wt, wts = ora.fp4_to_fp8_col(wp[row_token.numpy()], ws[row_token.numpy()], row_off.numpy())
    assert_bits_equal(u8(ft), wt, "col fp8")
    assert_bits_equal(to_f32_np(fts), wts, "col scales")


def test_moe_workload_full_size_sampled():
    """bf16 [32768, 7168] tokens routed top-8 to 256 experts (262144 rows):
    MXFP4 on sampled rows, the row form on sampled rows, the column form on
    sampled whole segments, all against the oracle."""
    m = fp4()
    T, H, E = 32768, 7168, 256
    x = workloads.moe_tokens(seed=0, tokens=T, hidden=H, device=dev())
    row_token, row_off = workloads.moe_routing(seed=0, tokens=T, experts=E)
    packed, scales = m.mxfp4_quantize(x)
    rng = np.random.default_rng(1)
    rows = np.concatenate([[0, T - 1], rng.integers(0, T, 30)])
    xs = to_f32_np(x[torch.from_numpy(rows).to(dev())])
    wp, ws = ora.mxfp4_quantize(xs)
    assert_bits_equal(u8(packed[torch.from_numpy(rows).to(dev())]), wp, "mxfp4 packed")
    assert_bits_equal(u8(scales[torch.from_numpy(rows).to(dev())]), ws, "mxfp4 scales")
    idx = row_token.to(dev())
    dp = packed.index_select(0, idx).contiguous()
    ds = scales.index_select(0, idx).contiguous()
    del x
    fp8, fsc = m.fp4_to_fp8_row(dp, ds)
    R = dp.shape[0]
    rs = torch.from_numpy(np.concatenate([[0, R - 1], rng.integers(0, R, 30)])).to(dev())
    wf, wfs = ora.fp4_to_fp8_row(u8(dp[rs]), u8(ds[rs]))
    assert_bits_equal(u8(fp8[rs]), wf, "row fp8")
    assert_bits_equal(to_f32_np(fsc[rs]), wfs, "row scales")
    del fp8, fsc
    segs = m.Segments(row_off, dev())
    ft, fts = m.fp4_to_fp8_col(dp, ds, segs)
    so = segs.scale_off_host.numpy()
    ro = row_off.numpy()
    sizes = np.diff(ro)
    pick = [int(np.argmax(sizes)), int(np.argmin(np.where(sizes > 0, sizes, 1 << 30))),
            E - 1] + list(rng.integers(0, E, 3))
    for e in pick:
        r0, n_e = int(ro[e]), int(sizes[e])
        if n_e == 0:
            continue
        wo, wsc = ora.fp4_to_fp8_col_segment(u8(dp[r0:r0 + n_e]), u8(ds[r0:r0 + n_e]), 0, n_e)
        got = u8(ft[H * r0:H * (r0 + n_e)]).reshape(H, n_e)
        assert_bits_equal(got, wo, f"col segment {e}")
        nb = (n_e + 127) // 128
        gs = to_f32_np(fts[H * int(so[e]):H * (int(so[e]) + nb)]).reshape(H, nb)
        assert_bits_equal(gs, wsc, f"col scales segment {e}")


# Segment layouts aimed at the column kernel's units, run with runs of 32
# token blocks (blocks are numbered across segments, ceil(n_e / 128) per
# segment):
#   - a segment that starts on a run's last block, so the next run begins
#     one block into it (that run first converts the segment's block 0, for
#     the carry and the row heads);
#   - one that starts two blocks before a run's end and ends inside the next
#     run (the next run converts block 0 for the heads and the block before
#     it for the carry);
#   - long segments across several runs; one-block segments of 31, 32, 33,
#     127, 128 and 129 tokens; empty segments between them.
RUN_LAYOUTS = [
    [31 * 128, 128 + 50, 7],
    [30 * 128, 3 * 128 + 5, 33, 0, 32],
    [29 * 128 + 1, 70 * 128 + 77, 31, 129],
    [127, 128, 129, 0, 31, 32, 33, 28 * 128 - 3, 40 * 128, 1, 300],
    [5000, 6000, 0, 4096, 4095, 4097],
]


@pytest.mark.parametrize("sizes", RUN_LAYOUTS)
@pytest.mark.parametrize("cols", [128, 384, 512])
@pytest.mark.parametrize("shift", [0, 13])
def test_fp4_to_fp8_col_run_boundaries(sizes, cols, shift):
    m = fp4()
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    rng = np.random.default_rng(R + cols + shift)
    packed = rng.integers(0, 256, (R, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (R, cols // 32), dtype=np.uint8)
    segs = m.Segments(torch.from_numpy(off), dev())
    pk = torch.from_numpy(packed).to(dev())
    sc = torch.from_numpy(scales).to(dev())
    out = torch.full((cols * R + 96,), 0xA5, dtype=torch.uint8, device=dev())
    n = cols * R
    m.fp4_to_fp8_col(pk, sc, segs, out[32 + shift:32 + shift + n], run_blocks=32)
    wo, _ = ora.fp4_to_fp8_col(packed, scales, off)
    o = u8(out)
    assert np.all(o[:32 + shift] == 0xA5) and np.all(o[32 + shift + n:] == 0xA5)
    assert_bits_equal(o[32 + shift:32 + shift + n], wo, f"fp8_t {sizes[:3]} {cols}")


@pytest.mark.parametrize("cols", [128, 384, 1152])
@pytest.mark.parametrize("shift", [0, 1, 7, 30])
def test_fp4_to_fp8_col_short_segments(cols, shift):
    """Segments of 1 .. 31 tokens, whose rows are too short for whole
    sectors: the kernel lays a CTA's rows out in order in shared memory and
    writes the span as whole sectors, its two partial ends byte by byte.
    Every length, empty segments and longer neighbours, feature groups of
    fewer than eight blocks (cols 128, 384, 1152), output offsets that put
    the span's start at several positions in a sector; against the oracle
    bit for bit, with canaries on both sides."""
    m = fp4()
    sizes = [0, 200] + list(range(1, 32)) + [0, 5, 0, 31, 140, 3]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    rng = np.random.default_rng(cols * 31 + shift)
    packed = rng.integers(0, 256, (R, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (R, cols // 32), dtype=np.uint8)
    segs = m.Segments(torch.from_numpy(off), dev())
    pk = torch.from_numpy(packed).to(dev())
    sc = torch.from_numpy(scales).to(dev())
    n = cols * R
    out = torch.full((n + 96,), 0x5A, dtype=torch.uint8, device=dev())
    fts = torch.empty(cols * segs.total_blocks, dtype=torch.float32, device=dev())
    m.fp4_to_fp8_col(pk, sc, segs, out[32 + shift:32 + shift + n], fts)
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    o = u8(out)
    assert np.all(o[:32 + shift] == 0x5A) and np.all(o[32 + shift + n:] == 0x5A)
    assert_bits_equal(o[32 + shift:32 + shift + n], wo, f"fp8_t short {cols} {shift}")
    assert_bits_equal(to_f32_np(fts), wsc, f"fp8_t scales short {cols} {shift}")


@pytest.mark.parametrize("nseg", [511, 512, 700])
def test_fp4_to_fp8_col_many_segments(nseg):
    """Up to 511 segments the kernel reads the segment offsets from a copy in
    shared memory, from 512 on from global memory: both paths, with a mix
    of empty, short, one-block and multi-block segments, against the oracle
    bit for bit (codes and scales)."""
    m = fp4()
    rng = np.random.default_rng(nseg)
    sizes = rng.choice([0, 1, 5, 31, 32, 33, 100, 128, 129, 300], nseg).tolist()
    sizes[nseg // 2] = 2000
    cols = 256
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    packed = rng.integers(0, 256, (R, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (R, cols // 32), dtype=np.uint8)
    segs = m.Segments(torch.from_numpy(off), dev())
    ft, fts = m.fp4_to_fp8_col(torch.from_numpy(packed).to(dev()),
                               torch.from_numpy(scales).to(dev()), segs)
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    assert_bits_equal(u8(ft), wo, f"fp8_t {nseg} segments")
    assert_bits_equal(to_f32_np(fts), wsc, f"fp8_t scales {nseg} segments")


@pytest.mark.parametrize("run", [0, 1, 2, 3, 7, 8, 29, 33, 40, 1000])
def test_fp4_to_fp8_col_any_run_length(run):
    """The column form does not depend on how the token blocks are cut into
    CTA work units: runs of 1 .. 1000 blocks (and the library's own choice,
    0) on segment layouts with long, one-block, short (< 32 tokens) and
    empty segments, against the oracle bit for bit, codes and scales, with
    the output at an odd byte offset."""
    m = fp4()
    rng = np.random.default_rng(run + 77)
    sizes = [31 * 128, 128 + 50, 7, 0, 29 * 128 + 1, 33, 128, 129, 300, 12, 4095, 5000, 1]
    sizes += rng.integers(0, 700, 12).tolist()
    cols = 384
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    packed = rng.integers(0, 256, (R, cols // 2), dtype=np.uint8)
    scales = rng.integers(110, 140, (R, cols // 32), dtype=np.uint8)
    segs = m.Segments(torch.from_numpy(off), dev())
    pk = torch.from_numpy(packed).to(dev())
    sc = torch.from_numpy(scales).to(dev())
    n = cols * R
    out = torch.full((n + 64,), 0xA5, dtype=torch.uint8, device=dev())
    fts = torch.empty(cols * segs.total_blocks, dtype=torch.float32, device=dev())
    m.fp4_to_fp8_col(pk, sc, segs, out[5:5 + n], fts, run_blocks=run)
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    o = u8(out)
    assert np.all(o[:5] == 0xA5) and np.all(o[5 + n:] == 0xA5)
    assert_bits_equal(o[5:5 + n], wo, f"fp8_t run {run}")
    assert_bits_equal(to_f32_np(fts), wsc, f"fp8_t scales run {run}")


@pytest.mark.parametrize("cols", [128, 384])
def test_fp4_to_fp8_full_range_scales(cols):
    """Row and column FP4 -> FP8 with UE8M0 bytes over their whole range
    0..255 (one block in eight at 0 or 255): shifts S_t - S_sub past 13 give
    zeros, and the fp32 output scales reach 2^-127 (subnormal) and 2^128
    (infinity).  Both forms against the oracle, bit for bit."""
    m = fp4()
    sizes = [300, 129, 0, 40, 1000]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    rng = np.random.default_rng(cols + 3)
    packed = rng.integers(0, 256, (R, cols // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (R, cols // 32), dtype=np.uint8)
    scales[rng.random(scales.shape) < 0.06] = 0
    scales[rng.random(scales.shape) < 0.06] = 255
    pk = torch.from_numpy(packed).to(dev())
    sc = torch.from_numpy(scales).to(dev())
    f8, f8s = m.fp4_to_fp8_row(pk, sc)
    wo, wsc = ora.fp4_to_fp8_row(packed, scales)
    assert_bits_equal(u8(f8), wo, "row fp8")
    assert_bits_equal(to_f32_np(f8s), wsc, "row scales")
    segs = m.Segments(torch.from_numpy(off), dev())
    ft, fts = m.fp4_to_fp8_col(pk, sc, segs)
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    assert_bits_equal(u8(ft), wo, "col fp8")
    assert_bits_equal(to_f32_np(fts), wsc, "col scales")
