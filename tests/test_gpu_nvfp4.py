"""GPU parity: NVFP4 amax / quantize / dequantize / qdq through the C ABI
against the CPU oracle, bit for bit (codes, scales, tensor scale, residual,
dequantized values, updated weights)."""
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


# sizes in elements: tiny, one CTA pass, several passes with a ragged tail
SIZES = [0, 16, 48, 4096, 16 * (256 * 7 + 37), 16 * 1216 * 256 * 2 + 16 * 5]


def _input(n, dtype, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(n, generator=g) * 0.02
    if n:
        k = max(1, n // 1000)
        idx = torch.randperm(n, generator=g)[:k]
        x[idx] = torch.randn(k, generator=g)
    return x.to(dtype).to(dev())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_quantize_compute_matches_oracle(dtype, n, rounding):
    if n > 100000 and rounding == "sr" and dtype == torch.float32:
        pytest.skip("covered by the bf16 case")
    m = fp4()
    x = _input(n, dtype, seed=n + 1)
    packed, scales, ts = m.nvfp4_quantize(x, rounding=rounding, seed=1234, step=7, tscale="compute")
    xn = to_f32_np(x)
    wp, ws, wt = ora.nvfp4_quantize(xn, rounding=ora.SR if rounding == "sr" else ora.RTN,
                                    seed=1234, step=7, tscale_mode=ora.TSCALE_COMPUTE)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    # dequantize, both output dtypes
    for od in (torch.float32, torch.bfloat16):
        y = m.nvfp4_dequantize(packed, scales, ts, (n,), od)
        wy = ora.nvfp4_dequantize(wp, ws, wt, n)
        if od == torch.bfloat16:
            assert_bits_equal(bf16_bits(y), ora.bf16_rn(wy), "dequant bf16")
        else:
            assert_bits_equal(to_f32_np(y), wy, "dequant f32")


@pytest.mark.parametrize("tscale", ["given", "from_amax"])
def test_quantize_tensor_scale_modes(tscale):
    m = fp4()
    n = 16 * 3000
    x = _input(n, torch.bfloat16, seed=5)
    xn = to_f32_np(x)
    if tscale == "given":
        ts_in = torch.full((1,), 0.00037, dtype=torch.float32, device=dev())
        packed, scales, ts = m.nvfp4_quantize(x, tscale="given", tensor_scale=ts_in)
        wp, ws, wt = ora.nvfp4_quantize(xn, tscale_mode=ora.TSCALE_GIVEN,
                                        tensor_scale=float(np.float32(0.00037)))
        assert ts.item() == np.float32(0.00037)  # GIVEN never writes
    else:
        amax = m.nvfp4_amax(x)
        assert np.float32(amax.item()) == np.float32(ora.nvfp4_amax(xn))
        packed, scales, ts = m.nvfp4_quantize(x, tscale="from_amax", amax_ws=amax)
        wp, ws, wt = ora.nvfp4_quantize(xn, tscale_mode=ora.TSCALE_COMPUTE)
        assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")


@pytest.mark.parametrize("given", [0.0, -1.0, float("inf"), float("nan")])
def test_given_scale_fallback_is_one(given):
    m = fp4()
    x = _input(16 * 64, torch.float32, seed=3)
    ts_in = torch.full((1,), given, dtype=torch.float32, device=dev())
    packed, scales, _ = m.nvfp4_quantize(x, tscale="given", tensor_scale=ts_in)
    wp, ws, _ = ora.nvfp4_quantize(to_f32_np(x), tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_error_feedback_residual_in_place(rounding, dtype):
    m = fp4()
    n = 16 * (256 * 3 + 11)
    x = _input(n, dtype, seed=9)
    g = torch.Generator(device="cpu").manual_seed(10)
    r0 = (torch.randn(n, generator=g) * 1e-3).to(torch.float32)
    r = r0.to(dev())
    packed, scales, ts = m.nvfp4_quantize(x, residual=r, rounding=rounding, seed=77, step=3)
    rn = r0.numpy().copy()
    wp, ws, wt = ora.nvfp4_quantize(to_f32_np(x), residual=rn,
                                    rounding=ora.SR if rounding == "sr" else ora.RTN,
                                    seed=77, step=3)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(to_f32_np(r), rn, "residual")


def test_worked_example_on_gpu():
    """hiren.me "Block scaling" worked block, through the CUDA path."""
    m = fp4()
    v = torch.zeros(16, dtype=torch.float32)
    v[:4] = torch.tensor([0.0132, -0.0471, -0.0109, -0.0347])
    ts = torch.ones(1, dtype=torch.float32, device=dev())
    packed, scales, _ = m.nvfp4_quantize(v.to(dev()), tscale="given", tensor_scale=ts)
    assert u8(packed)[:2].tolist() == [0xF3, 0xEB]
    assert u8(scales)[0] == 0x04
    y = m.nvfp4_dequantize(packed, scales, ts, (16,))
    assert y[:4].cpu().tolist() == [0.01171875, -0.046875, -0.01171875, -0.03125]


def test_degenerate_blocks():
    """All-zero blocks, a single nonzero, fp32 subnormals, negative zeros,
    values that saturate, and a huge dynamic range across blocks."""
    m = fp4()
    x = np.zeros(16 * 8, np.float32)
    x[16 + 3] = 1.0
    x[32:48] = np.float32(1e-40)                      # subnormals
    x[48:64] = -0.0
    x[64:80] = np.linspace(-3e38, 3e38, 16, dtype=np.float32)
    x[80:96] = np.float32(1e-30) * np.arange(16)
    x[96:112] = -np.float32(6.0)
    x[112:128] = np.float32(2.0 ** -140)
    xt = torch.from_numpy(x).to(dev())
    for mode in ("compute", "given"):
        ts = torch.ones(1, dtype=torch.float32, device=dev())
        packed, scales, tso = m.nvfp4_quantize(xt, tscale=mode, tensor_scale=ts)
        wp, ws, wt = ora.nvfp4_quantize(x, tscale_mode=ora.TSCALE_COMPUTE if mode == "compute"
                                        else ora.TSCALE_GIVEN, tensor_scale=1.0)
        assert np.float32(tso.item()) == np.float32(wt)
        assert_bits_equal(u8(packed), wp, f"packed {mode}")
        assert_bits_equal(u8(scales), ws, f"scales {mode}")
        y = m.nvfp4_dequantize(packed, scales, tso, (x.size,))
        assert_bits_equal(to_f32_np(y), ora.nvfp4_dequantize(wp, ws, wt, x.size), "dequant")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_infinite_inputs(rounding, dtype):
    """Blocks holding +-infinity among finite values, and blocks without
    one.  COMPUTE mode: the amax is infinite, so the tensor scale falls back
    to 1; GIVEN mode: a finite scale.  The block amax saturates the e4m3
    scale to 448, infinities encode as +-6 and the finite values beside them
    shrink; the other blocks are untouched.  Codes, scales and the
    dequantized values equal the oracle's."""
    m = fp4()
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(16 * 64) * 0.5).astype(np.float32)
    x[3] = np.inf
    x[16 * 5 + 7] = -np.inf
    x[16 * 9:16 * 10] = np.inf
    x[16 * 20 + 1] = np.inf
    x[16 * 20 + 2] = -np.inf
    xt = torch.from_numpy(x).to(dtype)
    xn = to_f32_np(xt)
    for mode, s_t in (("compute", 1.0), ("given", 0.01)):
        ts = torch.tensor([s_t], dtype=torch.float32, device=dev())
        packed, scales, tso = m.nvfp4_quantize(xt.to(dev()), rounding=rounding, seed=4, step=2,
                                               tscale=mode, tensor_scale=ts)
        wp, ws, wt = ora.nvfp4_quantize(xn, rounding=ora.SR if rounding == "sr" else ora.RTN,
                                        seed=4, step=2,
                                        tscale_mode=ora.TSCALE_COMPUTE if mode == "compute"
                                        else ora.TSCALE_GIVEN, tensor_scale=s_t)
        assert np.float32(tso.item()) == np.float32(wt), mode
        assert_bits_equal(u8(scales), ws, f"scales {mode}")
        assert_bits_equal(u8(packed), wp, f"packed {mode}")
        y = m.nvfp4_dequantize(packed, scales, tso, (x.size,))
        assert_bits_equal(to_f32_np(y), ora.nvfp4_dequantize(wp, ws, wt, x.size), f"y {mode}")


def test_empty_tensor_publishes_unit_scale():
    m = fp4()
    x = torch.empty(0, dtype=torch.float32, device=dev())
    ts = torch.full((1,), 5.0, device=dev())
    m.nvfp4_quantize(x, tscale="compute", tensor_scale=ts)
    assert ts.item() == 1.0


def test_nvfp4_roundtrip_workload_full():
    """The fp32 [1024, 1024] N(0, 0.02) + 0.1% N(0, 1) outlier workload, in
    full: amax, quantize (RTN, computed tensor scale), dequantize."""
    m = fp4()
    x = workloads.nvfp4_roundtrip(seed=0, device="cpu")
    xd = x.to(dev())
    packed, scales, ts = m.nvfp4_quantize(xd.view(-1))
    y = m.nvfp4_dequantize(packed, scales, ts, x.shape)
    wp, ws, wt = ora.nvfp4_quantize(x.numpy().ravel())
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(to_f32_np(y).ravel(), ora.nvfp4_dequantize(wp, ws, wt, x.numel()), "y")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
@pytest.mark.parametrize("with_g,with_r", [(True, True), (True, False), (False, True)])
def test_qdq_matches_oracle(rounding, with_g, with_r):
    m = fp4()
    n = 16 * (256 * 4 + 3)
    w0 = workloads.nvfp4_train_weight(seed=1, shape=(n // 16, 16), device="cpu").view(-1)
    g = workloads.nvfp4_train_grad(1, 0, shape=(n,), device="cpu") if with_g else None
    r0 = (torch.randn(n, generator=torch.Generator().manual_seed(2)) * 1e-4) if with_r else None
    w = w0.to(dev())
    rd = r0.to(dev()) if with_r else None
    gd = g.to(dev()) if with_g else None
    lr = 1e-4
    _, packed, scales, ts = m.nvfp4_qdq(w, gd, lr, rd, rounding=rounding, seed=5, step=11)
    wb = bf16_bits(w0).copy()
    rn = r0.numpy().copy() if with_r else None
    wp, ws, wt = ora.nvfp4_qdq(wb, None if g is None else g.numpy(), lr, rn,
                               rounding=ora.SR if rounding == "sr" else ora.RTN, seed=5, step=11)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(bf16_bits(w), wb, "W")
    if with_r:
        assert_bits_equal(to_f32_np(rd), rn, "residual")


@pytest.mark.parametrize("rounding", ["rtn", "sr"])
def test_qdq_infinite_gradient(rounding):
    """A training step whose gradient holds infinities (and one block of
    them): v = W - lr*G is infinite there, the amax too, so the tensor scale
    falls back to 1; those elements store +-6 * eff in W and an infinite
    residual.  W, residual, codes and scales equal the oracle's."""
    m = fp4()
    n = 16 * 200
    w0 = workloads.nvfp4_train_weight(seed=3, shape=(n // 64, 64), device="cpu").view(-1)
    g = workloads.nvfp4_train_grad(3, 0, shape=(n,), device="cpu").clone()
    g[7] = float("inf")
    g[16 * 50 + 3] = -float("inf")
    g[16 * 90:16 * 91] = float("inf")
    r0 = torch.randn(n, generator=torch.Generator().manual_seed(4)) * 1e-4
    w, rd = w0.to(dev()), r0.to(dev())
    _, packed, scales, ts = m.nvfp4_qdq(w, g.to(dev()), 1e-4, rd, rounding=rounding, seed=6,
                                        step=1)
    wb = bf16_bits(w0).copy()
    rn = r0.numpy().copy()
    wp, ws, wt = ora.nvfp4_qdq(wb, g.numpy(), 1e-4, rn,
                               rounding=ora.SR if rounding == "sr" else ora.RTN, seed=6, step=1)
    assert np.float32(ts.item()) == np.float32(wt) == np.float32(1.0)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(bf16_bits(w), wb, "W")
    assert_bits_equal(to_f32_np(rd), rn, "residual")


def test_qdq_training_workload_steps():
    """The bf16 [6144, 2048] N(0, 0.02) weight with G_t ~ N(0, 1), lr 1e-4,
    SR + error feedback: 3 full-size steps bit-exact, with the amax pass and
    the qdq pass as separate calls (FROM_AMAX) as the benchmark runs them."""
    m = fp4()
    shape = (6144, 2048)
    w0 = workloads.nvfp4_train_weight(seed=0, shape=shape, device="cpu")
    w = w0.to(dev()).view(-1)
    r = torch.zeros(w.numel(), dtype=torch.float32, device=dev())
    wb = bf16_bits(w0).ravel().copy()
    rn = np.zeros(w.numel(), np.float32)
    amax = torch.empty(1, dtype=torch.float32, device=dev())
    ts = torch.empty(1, dtype=torch.float32, device=dev())
    for t in range(3):
        g = workloads.nvfp4_train_grad(0, t, shape=shape, device="cpu").view(-1)
        gd = g.to(dev())
        m.nvfp4_qdq_amax(w, gd, 1e-4, r, amax_ws=amax)
        _, packed, scales, _ = m.nvfp4_qdq(w, gd, 1e-4, r, rounding="sr", seed=0, step=t,
                                           tscale="from_amax", amax_ws=amax, tensor_scale=ts)
        wp, ws, wt = ora.nvfp4_qdq(wb, g.numpy(), 1e-4, rn, rounding=ora.SR, seed=0, step=t)
        assert np.float32(ts.item()) == np.float32(wt)
        assert_bits_equal(bf16_bits(w), wb, f"W step {t}")
        assert_bits_equal(to_f32_np(r), rn, f"r step {t}")
        assert_bits_equal(u8(packed), wp, f"packed step {t}")
        assert_bits_equal(u8(scales), ws, f"scales step {t}")


def test_qdq_training_workload_100_steps_reduced():
    """The training configuration's 100 steps of W <- qdq(W - 1e-4 G) (SR +
    error feedback, a fresh gradient per step, the amax pass then the qdq
    pass) on a [256, 2048] slice-sized weight of the same distribution: W,
    the residual, the codes and the tensor scale equal the oracle's after
    every step."""
    m = fp4()
    shape = (256, 2048)
    w0 = workloads.nvfp4_train_weight(seed=3, shape=shape, device="cpu")
    w = w0.to(dev()).view(-1)
    r = torch.zeros(w.numel(), dtype=torch.float32, device=dev())
    wb = bf16_bits(w0).ravel().copy()
    rn = np.zeros(w.numel(), np.float32)
    amax = torch.empty(1, dtype=torch.float32, device=dev())
    ts = torch.empty(1, dtype=torch.float32, device=dev())
    for t in range(100):
        g = workloads.nvfp4_train_grad(3, t, shape=shape, device="cpu").view(-1)
        gd = g.to(dev())
        m.nvfp4_qdq_amax(w, gd, 1e-4, r, amax_ws=amax)
        _, packed, _, _ = m.nvfp4_qdq(w, gd, 1e-4, r, rounding="sr", seed=11, step=t,
                                      tscale="from_amax", amax_ws=amax, tensor_scale=ts)
        wp, _, wt = ora.nvfp4_qdq(wb, g.numpy(), 1e-4, rn, rounding=ora.SR, seed=11, step=t)
        assert np.float32(ts.item()) == np.float32(wt), t
        assert_bits_equal(u8(packed), wp, f"packed step {t}")
        assert_bits_equal(bf16_bits(w), wb, f"W step {t}")
        assert_bits_equal(to_f32_np(r), rn, f"r step {t}")


def test_qdq_sub_ulp_accumulation_on_gpu():
    """fp4-train "Correctness": a sub-ULP accumulation reaches 1.50 under EF
    and SR and stays at 0.50 under RTN (the same run as the oracle pin)."""
    m = fp4()
    blocks = 64
    w = torch.full((blocks, 16), 0.5)
    w[:, 0] = 6.0
    g = torch.full((blocks, 16), -(2.0 ** -7))
    g[:, 0] = 0.0
    ts = torch.ones(1, dtype=torch.float32, device=dev())
    out = {}
    for name, rounding, ef in (("rtn", "rtn", False), ("ef", "rtn", True), ("sr", "sr", False)):
        wd = w.to(torch.bfloat16).to(dev()).view(-1)
        gd = g.to(dev()).view(-1)
        r = torch.zeros(wd.numel(), device=dev()) if ef else None
        for t in range(128):
            m.nvfp4_qdq(wd, gd, 1.0, r, rounding=rounding, seed=0, step=t, tscale="given",
                        tensor_scale=ts, want_packed=False)
        out[name] = wd.view(blocks, 16)[:, 1:].float().cpu()
    assert torch.all(out["rtn"] == 0.5)
    assert torch.all(out["ef"] == 1.5)
    assert abs(out["sr"].mean().item() - 1.5) < 0.05


def test_qwen_shaped_matrices_sampled():
    """The Laplace weight set's matrix shapes at full size (one of each
    shape): tensor amax exact, then sampled blocks against the oracle."""
    m = fp4()
    rng = np.random.default_rng(0)
    for i, shape in enumerate([(1024, 4096), (4096, 12288)]):
        w = workloads.laplace_weight(100 + i, shape, device=dev())
        packed, scales, ts = m.nvfp4_quantize(w.view(-1))
        wn = to_f32_np(w).ravel()
        amax = ora.nvfp4_amax(wn)
        wt = ora.nvfp4_tensor_scale(amax)
        assert np.float32(ts.item()) == np.float32(wt)
        nb = wn.size // 16
        for b0 in list(rng.integers(0, nb - 64, 20)) + [0, nb - 64]:
            b0 = int(b0)
            wp, ws, _ = ora.nvfp4_blocks(wn[16 * b0:16 * (b0 + 64)], b0, wt)
            assert_bits_equal(u8(packed[8 * b0:8 * (b0 + 64)]), wp, f"packed {shape} @{b0}")
            assert_bits_equal(u8(scales[b0:b0 + 64]), ws, f"scales {shape} @{b0}")
        y = m.nvfp4_dequantize(packed, scales, ts, shape, torch.bfloat16)
        yb = bf16_bits(y).ravel()
        for b0 in rng.integers(0, nb - 64, 10):
            b0 = int(b0)
            wy = ora.nvfp4_dequantize(u8(packed[8 * b0:8 * (b0 + 64)]), u8(scales[b0:b0 + 64]),
                                      wt, 64 * 16)
            assert_bits_equal(yb[16 * b0:16 * (b0 + 64)], ora.bf16_rn(wy), "dequant bf16")


def test_rtn_quotients_on_and_near_rounding_midpoints():
    """Elements whose quotient v / scale lies exactly on, or within a few ulps
    of, an E2M1 rounding midpoint (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) and
    the saturation point, under many non-power-of-two decoded scales: the
    device's RTN codes must equal RN_e2m1(RN(v / scale)) (the oracle divides
    each element; the kernel's fast path must fall back exactly here)."""
    m = fp4()
    rng = np.random.default_rng(11)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    blocks = []
    s_t = np.float32(0.37)
    for _ in range(1200):
        bmax = np.float32(rng.uniform(0.05, 40.0))
        den6 = np.float32(6.0) * s_t
        sb = ora.e4m3_rn([np.float32(bmax / den6)])[0]
        eff = np.float32(np.float32(ora.e4m3_value([sb])[0]) * s_t)
        v = np.zeros(16, np.float32)
        v[0] = bmax
        for i in range(1, 16):
            mid = mids[rng.integers(0, mids.size)] * (1 if rng.random() < 0.5 else -1)
            base = np.float32(np.float32(mid) * eff)
            k = int(rng.integers(-3, 4))
            x = base
            step = np.float32(np.inf if k > 0 else -np.inf)
            for _ in range(abs(k)):
                x = np.nextafter(x, step)
            v[i] = x if abs(x) < bmax else base
        blocks.append(v)
    x = np.concatenate(blocks)
    ts = torch.full((1,), float(s_t), dtype=torch.float32, device=dev())
    packed, scales, _ = m.nvfp4_quantize(torch.from_numpy(x).to(dev()), tscale="given",
                                         tensor_scale=ts)
    wp, ws, _ = ora.nvfp4_quantize(x, tscale_mode=ora.TSCALE_GIVEN, tensor_scale=float(s_t))
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(u8(packed), wp, "packed")
    # the construction really produces quotients on midpoints
    eff_all = (ora.e4m3_value(ws).astype(np.float32) * s_t).astype(np.float32)
    q = (x.reshape(-1, 16) / eff_all[:, None]).astype(np.float32)
    assert np.isin(np.abs(q), mids[:-1]).sum() > 1000


def test_rtn_structural_ties_full_matrix():
    """bf16 weights under the computed tensor scale amax / (6 * 448) put many
    quotients v / scale exactly on E2M1 rounding midpoints (and some block
    maxima exactly on E4M3 midpoints); a whole 4M-element matrix is compared
    with the oracle, which divides every element."""
    m = fp4()
    w = workloads.laplace_weight(321, (1024, 4096), device=dev()).view(-1)
    packed, scales, ts = m.nvfp4_quantize(w)
    wn = to_f32_np(w)
    wp, ws, wt = ora.nvfp4_quantize(wn)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(u8(packed), wp, "packed")
    # the matrix really has exact ties (quotients equal to a midpoint)
    eff = (ora.e4m3_value(ws).astype(np.float32) * np.float32(wt)).astype(np.float32)
    q = (wn.reshape(-1, 16) / eff[:, None]).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    assert np.isin(np.abs(q), mids).sum() > 1000


@pytest.mark.parametrize("s_t", [2.0 ** -131, 2.0 ** 121])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_rtn_decoded_scale_outside_bracket_range(s_t, dtype):
    """A given tensor scale so small or so large that the decoded block
    scales fall outside [2^-125, 2^125], where the kernel cannot use its
    reciprocal bracket and every element of the block takes the exact
    division (all 16 elements of every lane go through the warp's pending
    list at once, many list flushes per pass)."""
    m = fp4()
    n = 16 * (256 * 5 + 7)
    g = torch.Generator(device="cpu").manual_seed(23)
    mag = torch.exp2(torch.randint(-6, 9, (n,), generator=g).float())
    # finite inputs only (NaN and Inf are outside the contract)
    x = (torch.randn(n, generator=g) * mag * float(s_t)).clamp(-3e38, 3e38).to(dtype)
    ts = torch.full((1,), s_t, dtype=torch.float32, device=dev())
    packed, scales, _ = m.nvfp4_quantize(x.to(dev()), tscale="given", tensor_scale=ts)
    wp, ws, _ = ora.nvfp4_quantize(to_f32_np(x), tscale_mode=ora.TSCALE_GIVEN,
                                   tensor_scale=float(np.float32(s_t)))
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(u8(packed), wp, "packed")
    eff = ora.e4m3_value(ws).astype(np.float64) * np.float32(s_t)
    out = (eff != 0) & ((eff < 2.0 ** -125) | (eff > 2.0 ** 125))
    assert out.mean() > 0.5


def test_rtn_error_feedback_on_structural_ties():
    """Round-to-nearest with error feedback on bf16 Laplace weights, whose
    quotients often sit exactly on E2M1 midpoints: blocks the kernel defers
    are redone from the untouched residual; codes, scales and residual are
    compared bit for bit."""
    m = fp4()
    w = workloads.laplace_weight(77, (512, 4096), device=dev()).view(-1)
    n = w.numel()
    r0 = (torch.randn(n, generator=torch.Generator().manual_seed(4)) * 1e-3).to(torch.float32)
    r = r0.to(dev())
    packed, scales, ts = m.nvfp4_quantize(w, residual=r, rounding="rtn")
    rn = r0.numpy().copy()
    wp, ws, wt = ora.nvfp4_quantize(to_f32_np(w), residual=rn, rounding=ora.RTN)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(to_f32_np(r), rn, "residual")


def test_rtn_qdq_on_structural_ties():
    """The in-place qdq step under round-to-nearest on bf16 Laplace weights
    (no gradient, no residual: v = W exactly, so quotients hit midpoints):
    deferred blocks are redone from the not yet updated W."""
    m = fp4()
    w0 = workloads.laplace_weight(78, (512, 4096), device="cpu").view(-1)
    w = w0.to(dev())
    _, packed, scales, ts = m.nvfp4_qdq(w, None, 0.0, None, rounding="rtn")
    wb = bf16_bits(w0).copy()
    wp, ws, wt = ora.nvfp4_qdq(wb, None, 0.0, None, rounding=ora.RTN)
    assert np.float32(ts.item()) == np.float32(wt)
    assert_bits_equal(u8(packed), wp, "packed")
    assert_bits_equal(u8(scales), ws, "scales")
    assert_bits_equal(bf16_bits(w), wb, "W")


def _nan_aware_equal(got_bits, want_f32, what):
    """bf16 bits against the oracle's fp32 values rounded to bf16: equal bit
    for bit, except that a NaN only has to be a NaN."""
    want = ora.bf16_rn(want_f32)
    got_nan = (got_bits & 0x7FFF) > 0x7F80
    want_nan = np.isnan(want_f32)
    assert np.array_equal(got_nan, want_nan), what
    assert_bits_equal(got_bits[~want_nan], want[~want_nan], what)


@pytest.mark.parametrize("s_t", [1.0, 0.000447591, 3.0e-41, 1.0e36])
def test_dequantize_every_code_and_scale_byte(s_t):
    """All 16 codes under all 256 scale bytes: the sign-set bytes (a negative
    decoded scale), 0x00 and 0x80 (zero), 0x7F and 0xFF (NaN).  A tensor
    scale of 1e36 overflows 448 * s_t; one of 3e-41 is subnormal.  bf16 and
    fp32 outputs, single-tensor and batched calls."""
    m = fp4()
    nb = 256 * 8 + 3  # every byte, eight times, and a ragged tail
    sc = np.concatenate([np.tile(np.arange(256, dtype=np.uint8), 8),
                         np.array([0x7E, 0x01, 0x80], np.uint8)])
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, nb * 8, dtype=np.uint8)
    codes[: 8 * 256] = np.tile(np.array([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE],
                                        np.uint8), 256)  # all 16 codes in every block
    pk = torch.from_numpy(codes).to(dev())
    sct = torch.from_numpy(sc).to(dev())
    ts = torch.tensor([s_t], dtype=torch.float32, device=dev())
    want = ora.nvfp4_dequantize(codes, sc, float(np.float32(s_t)), 16 * nb)
    yb = m.nvfp4_dequantize(pk, sct, ts, (16 * nb,), torch.bfloat16)
    _nan_aware_equal(bf16_bits(yb), want, "single bf16")
    yf = m.nvfp4_dequantize(pk, sct, ts, (16 * nb,), torch.float32)
    wn = np.isnan(want)
    assert np.array_equal(np.isnan(to_f32_np(yf)), wn)
    assert_bits_equal(to_f32_np(yf)[~wn], want[~wn], "single f32")
    # batched: the same blocks as three tensors (odd block counts)
    cuts = [0, 501, 1733, nb]
    pks = [pk[8 * a:8 * b].clone() for a, b in zip(cuts, cuts[1:])]
    scs = [sct[a:b].clone() for a, b in zip(cuts, cuts[1:])]
    for od in (torch.bfloat16, torch.float32):
        ys = [torch.full((16 * (b - a),), 7.0, dtype=od, device=dev())
              for a, b in zip(cuts, cuts[1:])]
        batch = m.Batch(packed=pks, scales=scs, ys=ys, sizes=[16 * (b - a) for a, b in
                                                               zip(cuts, cuts[1:])])
        m.nvfp4_dequantize_batched(batch, ts.repeat(3), od)
        for i, (a, b) in enumerate(zip(cuts, cuts[1:])):
            w = want[16 * a:16 * b]
            if od == torch.bfloat16:
                _nan_aware_equal(bf16_bits(ys[i]), w, f"batched bf16 {i}")
            else:
                g = to_f32_np(ys[i])
                assert np.array_equal(np.isnan(g), np.isnan(w))
                assert_bits_equal(g[~np.isnan(w)], w[~np.isnan(w)], f"batched f32 {i}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sr_on_and_near_the_rounding_thresholds(dtype):
    """Stochastic rounding where the quotient sits on, or one ulp from, the
    threshold lo + u * step that the element's own random word u defines
    (and on grid points, with zeros and saturating values): the kernel's
    division-free rule cannot decide these and must take the exact path.
    Each block holds a 6.0, so with a tensor scale of 1 its decoded scale is
    exactly 1 and the quotient is the element itself."""
    m = fp4()
    nb = 4096
    seed, step = 77, 5
    g = np.arange(16 * nb, dtype=np.uint64)
    u = (ora.rng_words(seed, step, g) >> 8).astype(np.float64) * 2.0 ** -24
    rng = np.random.default_rng(3)
    lo_tab = np.array([0, 0.5, 1, 1.5, 2, 3, 4], np.float64)
    step_tab = np.array([0.5, 0.5, 0.5, 0.5, 1, 1, 2], np.float64)
    c = rng.integers(0, 7, 16 * nb)
    a = lo_tab[c] + u * step_tab[c]                  # exactly on the threshold
    x = a.astype(np.float32)
    kind = rng.integers(0, 6, 16 * nb)
    x = np.where(kind == 1, np.nextafter(x, np.float32(np.inf)), x)
    x = np.where(kind == 2, np.nextafter(x, np.float32(0)), x)
    x = np.where(kind == 3, lo_tab[c].astype(np.float32), x)          # grid points
    x = np.where(kind == 4, np.float32(0.0), x)
    x = np.where(kind == 5, np.float32(5.99999), x)
    x = np.where(rng.integers(0, 2, 16 * nb) == 1, -x, x).astype(np.float32)
    x[::16] = 6.0
    xt = torch.from_numpy(x)
    if dtype == torch.bfloat16:
        xt = xt.to(torch.bfloat16)   # the thresholds move; still near-threshold cases
    one = torch.ones(1, device=dev())
    pk, sc, _ = m.nvfp4_quantize(xt.to(dev()), rounding="sr", seed=seed, step=step,
                                 tscale="given", tensor_scale=one)
    wp, ws, _ = ora.nvfp4_quantize(to_f32_np(xt), rounding=ora.SR, seed=seed, step=step,
                                   tscale_mode=ora.TSCALE_GIVEN, tensor_scale=1.0)
    assert_bits_equal(u8(sc), ws, "scales")
    assert_bits_equal(u8(pk), wp, "packed")
