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


def test_choose_schedule_follows_tiles_per_cta():
    """The rule on the three measured shapes (152 SMs): decode 1K/b32 and
    8K/b16 take the load-balanced split, the ragged 64-sequence full pool the
    chunked one; an empty batch takes the balanced split."""
    from fp8_paged_kv_append_gb300 import workloads
    from fp8_paged_kv_append_gb300.decode_step import choose_schedule
    assert choose_schedule(workloads.decode_1k_b32().seq_lens, 10, 152) == "balanced_fused"
    assert choose_schedule(workloads.decode_8k_b16().seq_lens, 10, 152) == "balanced_fused"
    assert choose_schedule(workloads.fullpool_layout(seed=4).seq_lens, 10, 152) == "fused"
    assert choose_schedule([0, 0], 10, 152) == "balanced_fused"
    # the boundary: exactly 160 tiles per CTA, then one page more
    assert choose_schedule([160 * 16 * 608 // 10], 10, 152) == "balanced_fused"
    assert choose_schedule([160 * 16 * 608 // 10 + 16], 10, 152) == "fused"
