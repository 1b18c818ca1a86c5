"""GPU parity: block scales in the blocked (swizzled) layout of block-scaled
tensor-core matmuls ([fp4-train] "Scope") -- the linear <-> blocked
conversions and the NVFP4 quantize that writes blocked scales directly --
against the CPU oracle, bit for bit.  The last tests pin the layout and the
nibble order to their consumer: torch._scaled_mm's NVFP4 matmul (cuBLASLt)
on operands made by the oracle, and on operands made by the CUDA path."""
import numpy as np
import pytest
import torch

import oracle as ora
from block_scaled_fp4_e2m1_gb300 import workloads
from parity_util import assert_bits_equal, dev, ensure_built, to_f32_np, u8

pytestmark = pytest.mark.gpu

GUARD = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def fp4():
    import block_scaled_fp4_e2m1_gb300 as m
    return m


# (rows, cols): 16-, 4- and 1-byte access paths, ragged row and column tiles,
# several units along a row (cols > 128), an empty matrix
SHAPES = [(1, 1), (128, 4), (129, 5), (300, 22), (5, 257), (1000, 3), (384, 64), (200, 160),
          (130, 272), (7, 400), (513, 132), (4096, 256), (3, 1030), (0, 9)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("offset", [0, 1, 4])
def test_to_and_from_blocked_match_oracle(rows, cols, offset):
    m = fp4()
    rng = np.random.default_rng(rows * 7919 + cols * 31 + offset)
    lin = rng.integers(0, 256, rows * cols, dtype=np.uint8)
    # the linear matrix starts `offset` bytes into its buffer (alignment paths)
    buf = torch.full((rows * cols + offset + GUARD,), 0x3C, dtype=torch.uint8, device=dev())
    buf[offset:offset + rows * cols] = torch.from_numpy(lin).to(dev())
    s = buf[offset:offset + rows * cols].view(rows, cols)
    size = m.fp4_blocked_scales_size(rows, cols)
    out = torch.full((size + GUARD,), 0xA5, dtype=torch.uint8, device=dev())
    m.fp4_scales_to_blocked(s, out=out[:size])
    assert_bits_equal(u8(out[:size]), ora.scales_to_blocked(lin, rows, cols), "blocked")
    assert (out[size:] == 0xA5).all()
    back = torch.full((rows * cols + offset + GUARD,), 0x5A, dtype=torch.uint8, device=dev())
    m.fp4_scales_from_blocked(out[:size], rows, cols,
                              out=back[offset:offset + rows * cols].view(rows, cols))
    assert_bits_equal(u8(back[offset:offset + rows * cols]), lin, "linear")
    assert (back[:offset] == 0x5A).all() and (back[offset + rows * cols:] == 0x5A).all()


def _inputs(rows, k, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, k, generator=g)
    # a power-of-two magnitude per 16-element block: block scales differ
    mag = torch.exp2(torch.randint(-3, 5, (rows, k // 16), generator=g).float())
    return (x * mag.repeat_interleave(16, dim=1)).to(dtype)


@pytest.mark.parametrize("rows,k", [(1, 16), (129, 80), (300, 352), (256, 4096), (1000, 48),
                                    (37, 2064)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding,with_res", [("rtn", False), ("sr", False), ("rtn", True),
                                               ("sr", True)])
def test_quantize_blocked_matches_oracle(rows, k, dtype, rounding, with_res):
    m = fp4()
    x = _inputs(rows, k, dtype, seed=rows * 13 + k)
    xn = to_f32_np(x).reshape(-1)
    res_np = (np.random.default_rng(5).standard_normal(xn.size).astype(np.float32) * 0.01
              if with_res else None)
    res = torch.from_numpy(res_np.copy()).to(dev()) if with_res else None
    size = m.fp4_blocked_scales_size(rows, k // 16)
    blk = torch.full((size + GUARD,), 0xA5, dtype=torch.uint8, device=dev())
    pk, _, ts = m.nvfp4_quantize_blocked(x.to(dev()), residual=res, rounding=rounding, seed=11,
                                         step=4, blocked_scales=blk[:size])
    wr = res_np.copy() if with_res else None
    wp, ws, wt = ora.nvfp4_quantize(xn, residual=wr, rounding=ora.SR if rounding == "sr"
                                    else ora.RTN, seed=11, step=4)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(pk).reshape(-1), wp, "packed")
    assert_bits_equal(u8(blk[:size]), ora.scales_to_blocked(ws, rows, k // 16), "blocked scales")
    assert (blk[size:] == 0xA5).all()
    if with_res:
        assert_bits_equal(to_f32_np(res), wr, "residual")


def test_quantize_blocked_given_scale_and_empty():
    m = fp4()
    x = _inputs(130, 96, torch.bfloat16, seed=3).to(dev())
    ts = torch.tensor([0.01], device=dev())
    pk, blk, _ = m.nvfp4_quantize_blocked(x, tscale="given", tensor_scale=ts)
    wp, ws, _ = ora.nvfp4_quantize(to_f32_np(x), tscale_mode=ora.TSCALE_GIVEN,
                                   tensor_scale=float(np.float32(0.01)))
    assert_bits_equal(u8(pk).reshape(-1), wp, "packed")
    assert_bits_equal(u8(blk), ora.scales_to_blocked(ws, 130, 6), "blocked")
    # an empty matrix still publishes its tensor scale (amax 0 -> 1)
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=dev())
    ts2 = torch.full((1,), -1.0, device=dev())
    m.nvfp4_quantize_blocked(e, tensor_scale=ts2)
    assert ts2.item() == 1.0


def test_quantize_blocked_weight_matrix_full_size():
    """A 12288 x 4096 bf16 Laplace weight (the gate/up projection shape): the
    fused blocked quantize equals the linear quantize followed by the
    conversion, and sampled tiles equal the oracle."""
    m = fp4()
    w = workloads.laplace_weight(77, (12288, 4096), device=dev())
    pk, blk, ts = m.nvfp4_quantize_blocked(w)
    p1, s1, t1 = m.nvfp4_quantize(w.view(-1))
    assert ts.item() == t1.item()
    assert torch.equal(pk.view(-1), p1)
    assert torch.equal(blk, m.fp4_scales_to_blocked(s1.view(12288, 256)))
    rng = np.random.default_rng(1)
    s_t = float(np.float32(ts.item()))
    for rt in [0, 95] + list(rng.integers(1, 95, 3)):
        rows = to_f32_np(w[128 * int(rt):128 * (int(rt) + 1)]).reshape(-1)
        _, ws, _ = ora.nvfp4_quantize(rows, tscale_mode=ora.TSCALE_GIVEN, tensor_scale=s_t)
        want = ora.scales_to_blocked(ws, 128, 256)
        got = u8(blk[int(rt) * 128 * 256:(int(rt) + 1) * 128 * 256])
        assert_bits_equal(got, want, f"row tile {rt}")


# ------------------------------------------------------ the consumer: a matmul

def _scaled_mm(a_codes, b_codes, a_blk, b_blk):
    """torch._scaled_mm's NVFP4 path: a [M, K/2] and b [N, K/2] packed E2M1
    with their e4m3 scales in the blocked layout; returns a @ b^T (bf16)."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this PyTorch has no float4_e2m1fn_x2")
    a = a_codes.view(torch.float4_e2m1fn_x2)
    b = b_codes.view(torch.float4_e2m1fn_x2)
    try:
        out = torch._scaled_mm(a, b.t(), a_blk.view(torch.float8_e4m3fn),
                               b_blk.view(torch.float8_e4m3fn), out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
    except (RuntimeError, NotImplementedError, TypeError) as e:
        pytest.skip(f"NVFP4 torch._scaled_mm is not available here: {str(e)[:200]}")
    return out.float().cpu().numpy().astype(np.float64)


def _dequant_np(packed, scales, n_rows, k):
    return ora.nvfp4_dequantize(packed, scales, 1.0, n_rows * k).astype(np.float64).reshape(n_rows, k)


def _check_product(got, a_deq, b_deq):
    ref = a_deq @ b_deq.T
    bound = np.abs(a_deq) @ np.abs(b_deq).T
    err = np.abs(got - ref)
    tol = 2.0 ** -8 * np.abs(ref) + 1e-4 * bound + 1e-30
    bad = np.nonzero(err > tol)
    assert bad[0].size == 0, (f"{bad[0].size} of {ref.size} products differ; first "
                              f"{[(int(i), int(j)) for i, j in zip(*bad)][:4]}: got "
                              f"{got[bad][:4]} want {ref[bad][:4]}")


@pytest.mark.parametrize("M,N,K", [(256, 128, 256), (328, 144, 352), (128, 256, 4096)])
def test_oracle_blocked_scales_feed_scaled_mm(M, N, K):
    """Operands quantized by the oracle (tensor scale 1), scales laid out by
    the oracle: the hardware product equals the exact product of the
    dequantized operands, so the layout and nibble order are the ones the
    tensor cores read."""
    a = to_f32_np(_inputs(M, K, torch.float32, seed=M + K)).reshape(-1)
    b = to_f32_np(_inputs(N, K, torch.float32, seed=N + 3 * K)).reshape(-1)
    ap, asc, _ = ora.nvfp4_quantize(a, tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    bp, bsc, _ = ora.nvfp4_quantize(b, tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    got = _scaled_mm(torch.from_numpy(ap).view(M, K // 2).to(dev()),
                     torch.from_numpy(bp).view(N, K // 2).to(dev()),
                     torch.from_numpy(ora.scales_to_blocked(asc, M, K // 16)).to(dev()),
                     torch.from_numpy(ora.scales_to_blocked(bsc, N, K // 16)).to(dev()))
    _check_product(got, _dequant_np(ap, asc, M, K), _dequant_np(bp, bsc, N, K))
    # a layout mistake is visible: the linear scales in place of the blocked
    # ones give a different product (same bytes, other places)
    if M % 128 == 0 and N % 128 == 0 and (K // 16) % 4 == 0:
        wrong = _scaled_mm(torch.from_numpy(ap).view(M, K // 2).to(dev()),
                           torch.from_numpy(bp).view(N, K // 2).to(dev()),
                           torch.from_numpy(asc).to(dev()), torch.from_numpy(bsc).to(dev()))
        assert not np.allclose(wrong, got, rtol=1e-2, atol=0)


def test_cuda_blocked_quantize_feeds_scaled_mm():
    """The CUDA path's own operands (nvfp4_quantize_blocked, tensor scale 1)
    give the same matmul as the oracle's."""
    m = fp4()
    M, N, K = 328, 144, 352
    a = _inputs(M, K, torch.bfloat16, seed=21).to(dev())
    b = _inputs(N, K, torch.bfloat16, seed=22).to(dev())
    one = torch.ones(1, device=dev())
    ap, ablk, _ = m.nvfp4_quantize_blocked(a, tscale="given", tensor_scale=one)
    bp, bblk, _ = m.nvfp4_quantize_blocked(b, tscale="given", tensor_scale=one)
    got = _scaled_mm(ap, bp, ablk, bblk)
    wap, was, _ = ora.nvfp4_quantize(to_f32_np(a), tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    wbp, wbs, _ = ora.nvfp4_quantize(to_f32_np(b), tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    _check_product(got, _dequant_np(wap, was, M, K), _dequant_np(wbp, wbs, N, K))


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_batched_blocked_matches_single_calls(rounding, dtype):
    """nvfp4_quantize_batched_blocked over matrices of assorted shapes (rows
    not a multiple of 128, k not a multiple of 64, one row, an empty
    matrix): every tensor's codes, blocked scales (padding included) and
    tensor scale equal nvfp4_quantize_blocked on it; guard bytes after each
    blocked buffer stay untouched; one tensor against the oracle."""
    m = fp4()
    shapes = [(1024, 512), (130, 48), (1, 16), (300, 352), (0, 64), (257, 2064)]
    xs = [_inputs(r, k, dtype, seed=40 + i).to(dev()) if r else
          torch.empty(0, k, dtype=dtype, device=dev()) for i, (r, k) in enumerate(shapes)]
    pks = [torch.full((r * k // 2,), 0x5A, dtype=torch.uint8, device=dev()) for r, k in shapes]
    sizes = [m.fp4_blocked_scales_size(r, k // 16) for r, k in shapes]
    bufs = [torch.full((sz + GUARD,), 0xA5, dtype=torch.uint8, device=dev()) for sz in sizes]
    blks = [b[:sz] for b, sz in zip(bufs, sizes)]
    batch = m.Batch(xs=[x.view(-1) for x in xs], packed=pks, scales=blks,
                    ks=[k for _, k in shapes])
    ts = m.nvfp4_quantize_batched_blocked(batch, dtype, rounding=rounding, seed=5, step=2,
                                          tscale="compute")
    for i, ((r, k), x) in enumerate(zip(shapes, xs)):
        p1, b1, t1 = m.nvfp4_quantize_blocked(x, rounding=rounding, seed=5, step=2)
        assert ts[i].item() == t1.item(), i
        assert_bits_equal(u8(pks[i]), u8(p1).reshape(-1), f"packed {i}")
        assert_bits_equal(u8(blks[i]), u8(b1), f"blocked {i}")
        assert (bufs[i][sizes[i]:] == 0xA5).all(), i
    r, k = shapes[5]
    wp, ws, wt = ora.nvfp4_quantize(to_f32_np(xs[5]).reshape(-1),
                                    rounding=ora.SR if rounding == "sr" else ora.RTN,
                                    seed=5, step=2)
    assert np.float32(ts[5].item()) == np.float32(wt)
    assert_bits_equal(u8(pks[5]), wp, "oracle packed")
    assert_bits_equal(u8(blks[5]), ora.scales_to_blocked(ws, r, k // 16), "oracle blocked")


@pytest.mark.parametrize("mode", ["given", "from_amax"])
def test_batched_blocked_tensor_scale_modes(mode):
    """The other two tensor-scale modes of the batched blocked quantize.
    given: per-tensor scales from the caller, among them 0 and NaN, which
    both quantizers replace by 1 (reading R6); from_amax: the scales follow
    from a preceding nvfp4_amax_batched.  Each tensor equals
    nvfp4_quantize_blocked on it under the same mode and scale."""
    m = fp4()
    shapes = [(256, 256), (130, 48), (64, 1024), (3, 16)]
    xs = [_inputs(r, k, torch.bfloat16, seed=70 + i).to(dev()) for i, (r, k) in enumerate(shapes)]
    pks = [torch.empty(r * k // 2, dtype=torch.uint8, device=dev()) for r, k in shapes]
    blks = [torch.empty(m.fp4_blocked_scales_size(r, k // 16), dtype=torch.uint8, device=dev())
            for r, k in shapes]
    batch = m.Batch(xs=[x.view(-1) for x in xs], packed=pks, scales=blks,
                    ks=[k for _, k in shapes])
    if mode == "given":
        given = [0.003, 0.0, float("nan"), 17.5]
        ts = torch.tensor(given, dtype=torch.float32, device=dev())
        m.nvfp4_quantize_batched_blocked(batch, torch.bfloat16, tscale="given", tensor_scale=ts)
        singles = [m.nvfp4_quantize_blocked(x, tscale="given",
                                            tensor_scale=torch.tensor([g], dtype=torch.float32,
                                                                      device=dev()))
                   for x, g in zip(xs, given)]
    else:
        amax = m.nvfp4_amax_batched(batch, torch.bfloat16)
        ts = m.nvfp4_quantize_batched_blocked(batch, torch.bfloat16, tscale="from_amax",
                                              amax=amax)
        singles = []
        for i, x in enumerate(xs):
            a1 = torch.zeros(1, dtype=torch.float32, device=dev())
            m.nvfp4_amax(x.view(-1), amax_ws=a1)
            assert a1.item() == amax[i].item(), i
            singles.append(m.nvfp4_quantize_blocked(x, tscale="from_amax", amax_ws=a1))
    for i, (p1, b1, t1) in enumerate(singles):
        if mode != "given":
            assert ts[i].item() == t1.item(), i
        assert_bits_equal(u8(pks[i]), u8(p1).reshape(-1), f"packed {i}")
        assert_bits_equal(u8(blks[i]), u8(b1), f"blocked {i}")
