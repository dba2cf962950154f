"""Host-side scale validation of the multi-layer decode step (no GPU)."""
import pytest
import torch

from fp8_paged_kv_append_gb300.decode_step import ScaleError, validate_scales


def test_validate_scales_accepts_positive_finite():
    validate_scales([torch.rand(10) + 0.01 for _ in range(3)])


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), 0.0, -1.0])
def test_validate_scales_rejects(bad):
    s = [torch.ones(10), torch.ones(10)]
    s[1][4] = bad
    with pytest.raises(ScaleError, match="layer 1"):
        validate_scales(s)
