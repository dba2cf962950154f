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


def _cpu_step(max_seq_len, schedule):
    from fp8_paged_kv_append_gb300.decode_step import MultiLayerDecode
    P, hkv = 8, 2
    kc = [torch.zeros((P, hkv, 16, 128), dtype=torch.float16)]
    vc = [torch.zeros((P, hkv, 16, 128), dtype=torch.uint8)]
    vs = [torch.ones(hkv)]
    bt = torch.zeros((2, 4), dtype=torch.int32)
    lens = torch.tensor([5, 9], dtype=torch.int32)
    slots = torch.zeros(2, dtype=torch.int64)
    return MultiLayerDecode(kc, vc, vs, bt, lens, slots, max_seq_len, 4 * hkv,
                            schedule=schedule)


def test_whole_schedule_is_one_launch_per_layer():
    """One CTA per (sequence, KV head) over the whole sequence: the split
    kernel writes the output, so a layer is one launch and the chunk covers
    the longest sequence."""
    step = _cpu_step(1000, "whole")
    assert step.launches_per_layer() == 1 and step.chunk == 1008


def test_whole_schedule_refuses_sequences_beyond_the_largest_chunk():
    with pytest.raises(ValueError, match="whole"):
        _cpu_step(9000, "whole")
