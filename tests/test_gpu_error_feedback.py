"""GPU parity: the keyed ErrorFeedback registry ([fp4-train] "Usage") against
the CPU oracle's qdq with an explicitly carried residual, bit for bit."""
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


@pytest.mark.parametrize("stochastic", [False, True])
def test_registry_qdq_matches_oracle_over_steps(stochastic):
    """Two keys, interleaved, five steps each: x_t = w + small drift; every
    returned weight and the final residuals equal the oracle's."""
    m = fp4()
    ef = m.ErrorFeedback(stochastic=stochastic, seed=7)
    rnd = ora.SR if stochastic else ora.RTN
    shapes = {"a": (64, 128), "b": (16, 256)}
    base = {k: workloads.nvfp4_train_weight(seed=i, shape=s, device="cpu").float()
            for i, (k, s) in enumerate(shapes.items())}
    res = {k: np.zeros(np.prod(s), np.float32) for k, s in shapes.items()}
    for t in range(5):
        for k in ("a", "b"):
            x = (base[k] + 1e-5 * (t + 1)).to(torch.bfloat16)
            got = ef.qdq(k, x.to(dev()), step=t)
            wb = bf16_bits(x).reshape(-1).copy()
            ora.nvfp4_qdq(wb, None, 0.0, res[k], rounding=rnd, seed=7, step=t)
            assert_bits_equal(bf16_bits(got).reshape(-1), wb, f"{k} step {t}")
    for k in shapes:
        assert_bits_equal(to_f32_np(ef.state_dict()[k]).reshape(-1), res[k], f"residual {k}")


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
    """A registry restored from another's state continues identically."""
    m = fp4()
    a = m.ErrorFeedback(seed=1)
    x = workloads.nvfp4_train_weight(seed=2, shape=(32, 64), device=dev())
    a.qdq("k", x, step=0)
    b = m.ErrorFeedback(seed=1)
    b.load_state_dict({k: v.clone() for k, v in a.state_dict().items()})
    ya, yb = a.qdq("k", x, step=1), b.qdq("k", x, step=1)
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
