"""GPU parity: the batched NVFP4 calls (one launch per pass over a list of
tensors) against the single-tensor calls on each tensor and against the CPU
oracle, bit for bit."""
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


# sizes in elements: empty, one block, ragged chunks, several chunks
SIZES = [16 * 4096 + 16 * 77, 0, 16, 16 * 255, 16 * 256, 16 * 257, 4096 * 1024 + 16 * 3, 16 * 999]


def _tensors(dtype, seed=0):
    out = []
    for i, n in enumerate(SIZES):
        g = torch.Generator().manual_seed(seed + i)
        x = torch.randn(n, generator=g) * (0.01 * (i + 1))
        if n:
            x[torch.randint(0, n, (max(1, n // 500),), generator=g)] *= 40
        out.append(x.to(dtype).to(dev()))
    return out


def _buffers(xs):
    pk = [torch.full((x.numel() // 2,), 0x5A, dtype=torch.uint8, device=dev()) for x in xs]
    sc = [torch.full((x.numel() // 16,), 0x5A, dtype=torch.uint8, device=dev()) for x in xs]
    return pk, sc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_batched_quantize_equals_single_calls(dtype, rounding):
    m = fp4()
    xs = _tensors(dtype)
    pk, sc = _buffers(xs)
    batch = m.Batch(xs=xs, packed=pk, scales=sc)
    assert batch.total_chunks == sum((n // 16 + 255) // 256 for n in SIZES)
    ts = m.nvfp4_quantize_batched(batch, dtype, rounding=rounding, seed=3, step=9,
                                  tscale="compute")
    for i, x in enumerate(xs):
        p1, s1, t1 = m.nvfp4_quantize(x, rounding=rounding, seed=3, step=9, tscale="compute")
        assert ts[i].item() == t1.item(), i
        assert_bits_equal(u8(pk[i]), u8(p1), f"packed {i}")
        assert_bits_equal(u8(sc[i]), u8(s1), f"scales {i}")
    # and against the oracle for two of them
    for i in (0, 6):
        wp, ws, wt = ora.nvfp4_quantize(to_f32_np(xs[i]), rounding=ora.SR if rounding == "sr"
                                        else ora.RTN, seed=3, step=9)
        assert np.float32(ts[i].item()) == np.float32(wt)
        assert_bits_equal(u8(pk[i]), wp, f"oracle packed {i}")
        assert_bits_equal(u8(sc[i]), ws, f"oracle scales {i}")


def test_batched_amax_and_modes():
    m = fp4()
    xs = _tensors(torch.bfloat16, seed=50)
    pk, sc = _buffers(xs)
    batch = m.Batch(xs=xs, packed=pk, scales=sc)
    amax = m.nvfp4_amax_batched(batch, torch.bfloat16)
    for i, x in enumerate(xs):
        assert np.float32(amax[i].item()) == np.float32(ora.nvfp4_amax(to_f32_np(x))), i
    # FROM_AMAX reuses it; GIVEN reads per-tensor scales and writes nothing
    ts = m.nvfp4_quantize_batched(batch, torch.bfloat16, tscale="from_amax", amax=amax)
    given = torch.tensor([0.001 * (i + 1) for i in range(len(xs))], device=dev())
    before = given.clone()
    pk2, sc2 = _buffers(xs)
    batch2 = m.Batch(xs=xs, packed=pk2, scales=sc2)
    m.nvfp4_quantize_batched(batch2, torch.bfloat16, tscale="given", tensor_scale=given)
    assert torch.equal(given, before)
    for i, x in enumerate(xs):
        p1, s1, t1 = m.nvfp4_quantize(x, tscale="compute")
        assert ts[i].item() == t1.item()
        assert_bits_equal(u8(pk[i]), u8(p1), f"from_amax {i}")
        g1 = given[i:i + 1].clone()
        p2, s2, _ = m.nvfp4_quantize(x, tscale="given", tensor_scale=g1)
        assert_bits_equal(u8(pk2[i]), u8(p2), f"given packed {i}")
        assert_bits_equal(u8(sc2[i]), u8(s2), f"given scales {i}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_batched_dequantize_equals_single_calls(out_dtype):
    m = fp4()
    xs = _tensors(torch.float32, seed=70)
    pk, sc = _buffers(xs)
    batch = m.Batch(xs=xs, packed=pk, scales=sc)
    ts = m.nvfp4_quantize_batched(batch, torch.float32, tscale="compute")
    ys = [torch.full((x.numel(),), -9.0, dtype=out_dtype, device=dev()) for x in xs]
    dbatch = m.Batch(packed=pk, scales=sc, ys=ys, sizes=[x.numel() for x in xs])
    m.nvfp4_dequantize_batched(dbatch, ts, out_dtype)
    for i in range(len(xs)):
        y1 = m.nvfp4_dequantize(pk[i], sc[i], ts[i:i + 1], (xs[i].numel(),), out_dtype)
        if out_dtype == torch.bfloat16:
            assert_bits_equal(bf16_bits(ys[i]), bf16_bits(y1), f"y {i}")
        else:
            assert_bits_equal(to_f32_np(ys[i]), to_f32_np(y1), f"y {i}")
    # scale NULL means 1
    m.nvfp4_dequantize_batched(dbatch, None, out_dtype)
    y1 = m.nvfp4_dequantize(pk[0], sc[0], None, (xs[0].numel(),), out_dtype)
    assert torch.equal(ys[0].view(torch.int16) if out_dtype == torch.bfloat16 else ys[0],
                       y1.view(torch.int16) if out_dtype == torch.bfloat16 else y1)


def test_batched_weight_set_layer_sampled():
    """One layer of the Qwen3-8B-shaped weight set (7 matrices) in one batch,
    sampled blocks against the oracle."""
    m = fp4()
    shapes = workloads.qwen3_8b_weight_shapes(layers=1)
    ws = [workloads.laplace_weight(200 + i, s, device=dev()).view(-1) for i, s in enumerate(shapes)]
    pk, sc = _buffers(ws)
    batch = m.Batch(xs=ws, packed=pk, scales=sc)
    ts = m.nvfp4_quantize_batched(batch, torch.bfloat16, tscale="compute")
    rng = np.random.default_rng(4)
    for i, w in enumerate(ws):
        wn = to_f32_np(w)
        wt = ora.nvfp4_tensor_scale(ora.nvfp4_amax(wn))
        assert np.float32(ts[i].item()) == np.float32(wt)
        nb = wn.size // 16
        for b0 in list(rng.integers(0, nb - 64, 6)) + [nb - 64]:
            b0 = int(b0)
            wp, wsc, _ = ora.nvfp4_blocks(wn[16 * b0:16 * (b0 + 64)], b0, wt)
            assert_bits_equal(u8(pk[i][8 * b0:8 * (b0 + 64)]), wp, f"packed {i} @{b0}")
            assert_bits_equal(u8(sc[i][b0:b0 + 64]), wsc, f"scales {i} @{b0}")


def test_batched_rtn_ties_and_extreme_scales_full():
    """A batch mixing tie-heavy bf16 Laplace matrices (computed scales) with
    tensors whose given scale puts the decoded block scales outside the
    kernel's bracket range: the per-warp list of pending elements then holds
    entries of several tensors at once.  Every tensor is compared in full
    with the oracle."""
    m = fp4()
    xs, given = [], []
    for i, s_t in enumerate([None, 2.0 ** -131, None, 2.0 ** 121, 0.37, None]):
        if s_t is None:
            x = workloads.laplace_weight(400 + i, (256, 1024 + 16 * i), device="cpu").view(-1)
            s = ora.nvfp4_tensor_scale(ora.nvfp4_amax(to_f32_np(x)))
        else:
            g = torch.Generator().manual_seed(500 + i)
            n = 16 * (256 * 3 + 5 * i)
            mag = torch.exp2(torch.randint(-6, 9, (n,), generator=g).float())
            x = (torch.randn(n, generator=g) * mag * s_t).clamp(-3e38, 3e38).to(torch.bfloat16)
            s = s_t
        xs.append(x.to(dev()))
        given.append(float(np.float32(s)))
    pk, sc = _buffers(xs)
    batch = m.Batch(xs=xs, packed=pk, scales=sc)
    ts = torch.tensor(given, dtype=torch.float32, device=dev())
    m.nvfp4_quantize_batched(batch, torch.bfloat16, tscale="given", tensor_scale=ts)
    for i, x in enumerate(xs):
        wp, ws, _ = ora.nvfp4_quantize(to_f32_np(x), tscale_mode=ora.TSCALE_GIVEN,
                                       tensor_scale=given[i])
        assert_bits_equal(u8(sc[i]), ws, f"scales {i}")
        assert_bits_equal(u8(pk[i]), wp, f"packed {i}")


def test_batched_full_weight_set_sampled():
    """The whole 36-layer Qwen3-8B-shaped weight set (252 bf16 matrices,
    6.95 G weights) through the launches the benchmark times: one batched
    amax, one batched quantize (tensor scales from that amax) and one batched
    dequantize.  Every tensor scale against the oracle's, sampled blocks of
    every matrix against the oracle bit for bit."""
    m = fp4()
    shapes = workloads.qwen3_8b_weight_shapes(layers=36)
    mats = [workloads.laplace_weight(100 + i, s, device=dev()).view(-1)
            for i, s in enumerate(shapes)]
    pks = [torch.empty(w.numel() // 2, dtype=torch.uint8, device=dev()) for w in mats]
    scs = [torch.empty(w.numel() // 16, dtype=torch.uint8, device=dev()) for w in mats]
    ys = [torch.empty(w.numel(), dtype=torch.bfloat16, device=dev()) for w in mats]
    qb = m.Batch(xs=mats, packed=pks, scales=scs)
    db = m.Batch(packed=pks, scales=scs, ys=ys, sizes=[w.numel() for w in mats])
    am = m.nvfp4_amax_batched(qb, torch.bfloat16)
    ts = m.nvfp4_quantize_batched(qb, torch.bfloat16, tscale="from_amax", amax=am)
    m.nvfp4_dequantize_batched(db, ts, torch.bfloat16)
    rng = np.random.default_rng(36)
    ts_h = ts.cpu().numpy()
    for i, w in enumerate(mats):
        nb = w.numel() // 16
        # the oracle's amax over the whole matrix, on the host
        wt = ora.nvfp4_tensor_scale(ora.nvfp4_amax(to_f32_np(w)))
        assert np.float32(ts_h[i]) == np.float32(wt), i
        for b0 in [0, nb - 32, int(rng.integers(0, nb - 32))]:
            v = to_f32_np(w[16 * b0:16 * (b0 + 32)])
            wp, wsc, wq = ora.nvfp4_blocks(v, b0, wt)
            assert_bits_equal(u8(pks[i][8 * b0:8 * (b0 + 32)]), wp, f"packed {i} @{b0}")
            assert_bits_equal(u8(scs[i][b0:b0 + 32]), wsc, f"scales {i} @{b0}")
            assert_bits_equal(bf16_bits(ys[i][16 * b0:16 * (b0 + 32)]), ora.bf16_rn(wq),
                              f"dequant {i} @{b0}")
    del mats, pks, scs, ys
    torch.cuda.empty_cache()
