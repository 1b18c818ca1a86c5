"""GPU parity under randomized stress: many seeded configurations of NVFP4
quantize / dequantize / qdq, single-tensor, blocked-scale and batched, with
mixed magnitudes, exact ties, zeros, subnormals and near-saturating values,
against the CPU oracle, bit for bit.  Each trial is small; together they
walk the division-free fast paths (certified brackets, tie rule, the SR
threshold rule) through many scale regimes."""
import numpy as np
import pytest
import torch

import oracle as ora
from parity_util import assert_bits_equal, bf16_bits, dev, ensure_built, to_f32_np, u8

pytestmark = pytest.mark.gpu

TRIALS = 160


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def fp4():
    import block_scaled_fp4_e2m1_gb300 as m
    return m


def _stress(rng, n):
    """n values (n % 16 == 0): per-block magnitudes over 2^-40 .. 2^40, some
    blocks of exact grid multiples (ties under power-of-two scales), zeros,
    subnormal-scale values and single large outliers."""
    nb = n // 16
    mag = np.exp2(rng.integers(-40, 41, nb)).astype(np.float64)
    x = rng.standard_normal((nb, 16)) * mag[:, None]
    kind = rng.integers(0, 8, nb)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5])
    x[kind == 1] = (rng.choice(grid, (int((kind == 1).sum()), 16)) *
                    rng.choice([-1, 1], (int((kind == 1).sum()), 16)) *
                    mag[kind == 1][:, None])
    x[kind == 2] = 0.0
    x[kind == 3] *= 2.0 ** -100
    x[kind == 4, 0] *= 1000.0
    x = x.reshape(-1)
    return np.clip(x, -1e37, 1e37).astype(np.float32)


def _case(trial):
    rng = np.random.default_rng(9000 + trial)
    n = 16 * int(rng.integers(1, 6000))
    dtype = torch.bfloat16 if trial % 2 == 0 else torch.float32
    x = torch.from_numpy(_stress(rng, n)).to(dtype)
    rounding = "sr" if trial % 3 == 0 else "rtn"
    mode = ("given", "compute")[trial % 4 == 1]
    s_t = float(np.float32(2.0 ** float(rng.integers(-60, 40)) * rng.uniform(0.5, 2.0)))
    with_res = trial % 5 == 2
    return rng, n, dtype, x, rounding, mode, s_t, with_res


@pytest.mark.parametrize("trial", range(TRIALS))
def test_fuzz_quantize_dequantize(trial):
    m = fp4()
    rng, n, dtype, x, rounding, mode, s_t, with_res = _case(trial)
    xn = to_f32_np(x)
    res_np = (rng.standard_normal(n).astype(np.float32) * np.float32(2.0 ** -10)
              if with_res else None)
    ts = torch.tensor([s_t], dtype=torch.float32, device=dev())
    res = torch.from_numpy(res_np.copy()).to(dev()) if with_res else None
    pk, sc, t = m.nvfp4_quantize(x.to(dev()), residual=res, rounding=rounding, seed=trial,
                                 step=trial * 7, tscale=mode, tensor_scale=ts)
    wr = res_np.copy() if with_res else None
    wp, ws, wt = ora.nvfp4_quantize(xn, residual=wr, rounding=ora.SR if rounding == "sr"
                                    else ora.RTN, seed=trial, step=trial * 7,
                                    tscale_mode=ora.TSCALE_GIVEN if mode == "given"
                                    else ora.TSCALE_COMPUTE, tensor_scale=s_t)
    assert np.float32(t.item()) == np.float32(wt), trial
    assert_bits_equal(u8(sc), ws, f"scales {trial}")
    assert_bits_equal(u8(pk), wp, f"packed {trial}")
    if with_res:
        assert_bits_equal(to_f32_np(res), wr, f"residual {trial}")
    wy = ora.nvfp4_dequantize(wp, ws, wt, n)
    y = m.nvfp4_dequantize(pk, sc, t, (n,), torch.bfloat16)
    ok = np.isfinite(wy)
    assert_bits_equal(bf16_bits(y)[ok], ora.bf16_rn(wy)[ok], f"dequant {trial}")


@pytest.mark.parametrize("trial", range(0, TRIALS, 3))
def test_fuzz_blocked_and_batched(trial):
    """The same stress as matrices: the blocked-scale quantize against the
    oracle's scales laid out, and a batch of the trial's tensor with two
    others against the single-tensor results."""
    m = fp4()
    rng, n, dtype, x, rounding, mode, s_t, _ = _case(trial)
    k = 16 * int(rng.integers(1, 9))
    rows = n // k
    xm = x[: rows * k].view(rows, k)
    ts = torch.tensor([s_t], dtype=torch.float32, device=dev())
    pk, blk, t = m.nvfp4_quantize_blocked(xm.to(dev()), rounding=rounding, seed=trial, step=1,
                                          tscale=mode, tensor_scale=ts.clone())
    wp, ws, wt = ora.nvfp4_quantize(to_f32_np(xm).reshape(-1),
                                    rounding=ora.SR if rounding == "sr" else ora.RTN,
                                    seed=trial, step=1,
                                    tscale_mode=ora.TSCALE_GIVEN if mode == "given"
                                    else ora.TSCALE_COMPUTE, tensor_scale=s_t)
    assert_bits_equal(u8(pk).reshape(-1), wp, f"blocked packed {trial}")
    assert_bits_equal(u8(blk), ora.scales_to_blocked(ws, rows, k // 16), f"blocked {trial}")
    others = [torch.from_numpy(_stress(rng, 16 * int(rng.integers(1, 3000)))).to(dtype)
              for _ in range(2)]
    xs = [x.to(dev())] + [o.to(dev()) for o in others]
    pks = [torch.empty(v.numel() // 2, dtype=torch.uint8, device=dev()) for v in xs]
    scs = [torch.empty(v.numel() // 16, dtype=torch.uint8, device=dev()) for v in xs]
    batch = m.Batch(xs=xs, packed=pks, scales=scs)
    tss = m.nvfp4_quantize_batched(batch, dtype, rounding=rounding, seed=trial, step=2,
                                   tscale="compute")
    for i, v in enumerate(xs):
        p1, s1, t1 = m.nvfp4_quantize(v, rounding=rounding, seed=trial, step=2, tscale="compute")
        assert tss[i].item() == t1.item()
        assert_bits_equal(u8(pks[i]), u8(p1), f"batched packed {trial}.{i}")
        assert_bits_equal(u8(scs[i]), u8(s1), f"batched scales {trial}.{i}")


@pytest.mark.parametrize("trial", range(0, TRIALS, 4))
def test_fuzz_qdq(trial):
    """The fused training step on stressed bf16 weights with a gradient and
    a residual, RTN and SR."""
    m = fp4()
    rng = np.random.default_rng(7000 + trial)
    n = 16 * int(rng.integers(1, 4000))
    w = torch.from_numpy(_stress(rng, n)).to(torch.bfloat16)
    gr = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 5))).astype(np.float32)
    r0 = (rng.standard_normal(n) * 2.0 ** -12).astype(np.float32)
    rounding = "sr" if trial % 8 == 0 else "rtn"
    wd = w.clone().to(dev())
    rd = torch.from_numpy(r0.copy()).to(dev())
    m.nvfp4_qdq(wd, torch.from_numpy(gr).to(dev()), 1e-3, rd, rounding=rounding, seed=trial,
                step=3, tscale="compute")
    wb = bf16_bits(w).copy()
    rn = r0.copy()
    ora.nvfp4_qdq(wb, gr, 1e-3, rn, rounding=ora.SR if rounding == "sr" else ora.RTN,
                  seed=trial, step=3)
    assert_bits_equal(bf16_bits(wd), wb, f"qdq W {trial}")
    assert_bits_equal(to_f32_np(rd), rn, f"qdq residual {trial}")


@pytest.mark.parametrize("trial", range(16))
def test_fuzz_fp4_to_fp8_col(trial):
    """FP4RowToFP8Col on random ragged segment sets: empty, tiny (rows under
    32 bytes), medium and long segments (crossing several 32-block runs), an
    output that starts at a random byte offset, canaries around it."""
    m = fp4()
    rng = np.random.default_rng(5000 + trial)
    cols = int(rng.choice([128, 256, 384]))
    nseg = int(rng.integers(1, 40))
    kinds = rng.integers(0, 4, nseg)
    sizes = np.where(kinds == 0, 0, np.where(kinds == 1, rng.integers(1, 32, nseg),
                     np.where(kinds == 2, rng.integers(32, 700, nseg),
                              rng.integers(700, 6000, nseg))))
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    R = int(off[-1])
    packed = rng.integers(0, 256, (max(R, 1), cols // 2), dtype=np.uint8)[:R]
    scales = rng.integers(110, 140, (max(R, 1), cols // 32), dtype=np.uint8)[:R]
    segs = m.Segments(torch.from_numpy(off), dev())
    pk = torch.from_numpy(np.ascontiguousarray(packed)).to(dev())
    sc = torch.from_numpy(np.ascontiguousarray(scales)).to(dev())
    shift = int(rng.integers(0, 16))
    out = torch.full((cols * R + 96,), 0xA5, dtype=torch.uint8, device=dev())
    osc = torch.full((cols * segs.total_blocks + 16,), -7.0, dtype=torch.float32, device=dev())
    m.fp4_to_fp8_col(pk, sc, segs, out[32 + shift:32 + shift + cols * R],
                     osc[8:8 + cols * segs.total_blocks])
    wo, wsc = ora.fp4_to_fp8_col(packed, scales, off)
    o = u8(out)
    assert np.all(o[:32 + shift] == 0xA5) and np.all(o[32 + shift + cols * R:] == 0xA5)
    assert_bits_equal(o[32 + shift:32 + shift + cols * R], wo, f"fp8_t {trial}")
    s = to_f32_np(osc)
    assert np.all(s[:8] == -7.0) and np.all(s[8 + cols * segs.total_blocks:] == -7.0)
    assert_bits_equal(s[8:8 + cols * segs.total_blocks], wsc, f"fp8_t scales {trial}")
