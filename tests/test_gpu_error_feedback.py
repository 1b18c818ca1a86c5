"""GPU parity: the keyed ErrorFeedback registry ([fp4-train] "Usage": a
residual per weight, carried into the next quantization) against the CPU
oracle with an explicitly carried residual, bit for bit.  bf16 inputs take
the fused qdq; fp32 inputs take quantize-with-residual plus dequantize, so
that parts of x below bf16 resolution still reach the residual
([fp4-train] "Correctness": sub-ULP updates accumulate instead of
stalling)."""
import numpy as np
import pytest
import torch

import oracle as ora
from block_scaled_fp4_e2m1_gb300 import workloads
from parity_util import assert_bits_equal, bf16_bits, dev, ensure_built, to_f32_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def fp4():
    import block_scaled_fp4_e2m1_gb300 as m
    return m


def oracle_registry_step(x, r, rnd, seed, step):
    """The oracle's error-feedback round trip of fp32 x with residual r (in
    place): bf16 bits of dequant(quantize(x + r))."""
    pk, sc, ts = ora.nvfp4_quantize(x, residual=r, rounding=rnd, seed=seed, step=step)
    return ora.bf16_rn(ora.nvfp4_dequantize(pk, sc, ts, x.size))


@pytest.mark.parametrize("stochastic", [False, True])
def test_registry_qdq_bf16_matches_oracle_over_steps(stochastic):
    """Two keys, interleaved, five steps each, bf16 inputs x_t = w + 1e-3 (t+1)
    (a drift of several bf16 ulps, so every step's input differs); every
    returned weight and the final residuals equal the oracle's qdq."""
    m = fp4()
    ef = m.ErrorFeedback(stochastic=stochastic, seed=7)
    rnd = ora.SR if stochastic else ora.RTN
    shapes = {"a": (64, 128), "b": (16, 256)}
    base = {k: workloads.nvfp4_train_weight(seed=i, shape=s, device="cpu").float()
            for i, (k, s) in enumerate(shapes.items())}
    res = {k: np.zeros(np.prod(s), np.float32) for k, s in shapes.items()}
    prev = {}
    for t in range(5):
        for k in ("a", "b"):
            x = (base[k] + 1e-3 * (t + 1)).to(torch.bfloat16)
            if k in prev:  # the drift is representable: the input really moves
                assert (bf16_bits(x) != prev[k]).mean() > 0.9
            prev[k] = bf16_bits(x)
            got = ef.qdq(k, x.to(dev()), step=t)
            wb = bf16_bits(x).reshape(-1).copy()
            ora.nvfp4_qdq(wb, None, 0.0, res[k], rounding=rnd, seed=7, step=t)
            assert_bits_equal(bf16_bits(got).reshape(-1), wb, f"{k} step {t}")
    for k in shapes:
        assert_bits_equal(to_f32_np(ef.state_dict()[k]).reshape(-1), res[k], f"residual {k}")


@pytest.mark.parametrize("stochastic", [False, True])
def test_registry_qdq_fp32_below_bf16_resolution(stochastic):
    """fp32 x_t = w + d_t with |d_t| below half a bf16 ulp of w, 12 steps: the
    registry equals the oracle's quantize-with-residual + dequantize bit for
    bit (returned bf16 values and residuals), and the residuals differ from
    those of the bf16-rounded inputs, which would drop d_t."""
    m = fp4()
    ef = m.ErrorFeedback(stochastic=stochastic, seed=11)
    rnd = ora.SR if stochastic else ora.RTN
    w = workloads.nvfp4_train_weight(seed=3, shape=(64, 128), device="cpu")
    wn = w.float().numpy().ravel()
    half_ulp = np.ldexp(np.float32(1.0), np.frexp(np.abs(wn) + 1e-30)[1] - 9).astype(np.float32)
    rng = np.random.default_rng(5)
    r = np.zeros(wn.size, np.float32)
    r_bf16 = np.zeros(wn.size, np.float32)
    for t in range(12):
        d = (rng.uniform(-0.45, 0.45, wn.size) * half_ulp).astype(np.float32)
        x = (wn + d).astype(np.float32)
        assert np.array_equal(ora.bf16_rn(x), bf16_bits(w).ravel())  # bf16 would drop d
        got = ef.qdq("w", torch.from_numpy(x).view(64, 128).to(dev()), step=t)
        want = oracle_registry_step(x, r, rnd, 11, t)
        assert_bits_equal(bf16_bits(got).reshape(-1), want, f"step {t}")
        oracle_registry_step(ora.bf16_to_f32(ora.bf16_rn(x)), r_bf16, rnd, 11, t)
    assert_bits_equal(to_f32_np(ef.state_dict()["w"]).reshape(-1), r, "residual")
    assert (r != r_bf16).mean() > 0.5


def test_registry_sub_ulp_accumulation_fp32():
    """[fp4-train] "Correctness" through the registry with fp32 inputs: a
    block of 15 weights at 0.5 (anchor 6.0 keeps the decoded block scale at
    exactly 1 under the computed tensor scale) gets x_t = w_t + 2^-10, an
    update below half a bf16 ulp of 0.5.  After 1024 RTN + error-feedback
    steps every weight is exactly 1.5 (q + r = 0.5 + t 2^-10 holds exactly),
    and every step equals the oracle's."""
    m = fp4()
    ef = m.ErrorFeedback(seed=0)
    d = np.float32(2.0 ** -10)
    wv = np.full(16, 0.5, np.float32)
    wv[0] = 6.0
    r = np.zeros(16, np.float32)
    assert ora.bf16_rn(np.float32(0.5) + d) == ora.bf16_rn(np.float32(0.5))
    for t in range(1024):
        x = wv.copy()
        x[1:] += d
        got = ef.qdq("k", torch.from_numpy(x).to(dev()), step=t)
        want = oracle_registry_step(x, r, ora.RTN, 0, t)
        assert_bits_equal(bf16_bits(got), want, f"step {t}")
        wv = ora.bf16_to_f32(want)
    assert wv[0] == 6.0 and np.all(wv[1:] == 1.5)


def test_registry_fused_step_matches_oracle():
    """step(): W <- qdq((W - lr*G) + r) in place, three steps."""
    m = fp4()
    ef = m.ErrorFeedback(stochastic=True, seed=3)
    w0 = workloads.nvfp4_train_weight(seed=5, shape=(96, 64), device="cpu").view(-1)
    w = w0.to(dev())
    wb = bf16_bits(w0).copy()
    r = np.zeros(w0.numel(), np.float32)
    for t in range(3):
        g = workloads.nvfp4_train_grad(5, t, shape=(w0.numel(),), device="cpu")
        ef.step("w", w, g.to(dev()), 1e-3, step=t)
        ora.nvfp4_qdq(wb, g.numpy(), 1e-3, r, rounding=ora.SR, seed=3, step=t)
        assert_bits_equal(bf16_bits(w), wb, f"step {t}")
    assert_bits_equal(to_f32_np(ef.residual("w", w)), r, "residual")


def test_registry_state_round_trip():
    """A registry restored from another's state continues identically, for a
    bf16 and an fp32 key."""
    m = fp4()
    a = m.ErrorFeedback(seed=1)
    x = workloads.nvfp4_train_weight(seed=2, shape=(32, 64), device=dev())
    xf = x.float() + 1e-6
    a.qdq("k", x, step=0)
    a.qdq("f", xf, step=0)
    b = m.ErrorFeedback(seed=1)
    b.load_state_dict({k: v.clone() for k, v in a.state_dict().items()})
    for key, inp in (("k", x), ("f", xf)):
        ya, yb = a.qdq(key, inp, step=1), b.qdq(key, inp, step=1)
        assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
