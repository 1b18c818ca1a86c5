"""Host-side bookkeeping of the ErrorFeedback registry (CPU, no kernel call)."""
import pytest
import torch

from block_scaled_fp4_e2m1_gb300 import ErrorFeedback


def test_residuals_are_created_once_per_key_and_checked():
    ef = ErrorFeedback()
    w = torch.zeros(4, 16)
    r = ef.residual("a", w)
    assert r.dtype == torch.float32 and r.shape == w.shape and not r.any()
    assert ef.residual("a", w) is r
    with pytest.raises(ValueError):
        ef.residual("a", torch.zeros(8, 16))
    ef.residual("b", torch.zeros(16))
    assert sorted(ef.keys()) == ["a", "b"]
    ef.reset("a")
    assert ef.keys() == ["b"]
    ef.reset()
    assert ef.keys() == []


def test_state_dict_requires_fp32():
    ef = ErrorFeedback(stochastic=True, seed=3)
    assert ef.rounding == "sr" and ef.seed == 3
    with pytest.raises(ValueError):
        ef.load_state_dict({"a": torch.zeros(16, dtype=torch.bfloat16)})
    ef.load_state_dict({"a": torch.ones(16)})
    assert torch.equal(ef.state_dict()["a"], torch.ones(16))
