"""Full-pool ragged decode across 40 layers (32 GiB of K16/V8 pools, 223,696
slots per layer, batch 64 with lengths in [1, 8192]) through the graph-captured
multi-layer step, checked against the oracle on every sequence of layers 0,
17 and 39.  The pools are drawn on the device with torch; those layers' pools
are copied to the host before any kernel runs, and the oracle appends the new
tokens itself, so no oracle input comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_append_gb300 import workloads
from cases import check_close, dev, to_dev

pytestmark = pytest.mark.gpu

LAYERS = 40
CHECKED_LAYERS = (0, 17, 39)


@pytest.fixture(scope="module")
def setup():
    from fp8_paged_kv_append_gb300 import k16v8 as K
    from fp8_paged_kv_append_gb300.decode_step import MultiLayerDecode
    K.load_library()
    lay = workloads.fullpool_layout(seed=4)
    P, B = lay.num_pages, len(lay.seq_lens)
    assert P * 16 == 223696 and int(np.sum(-(-lay.seq_lens // 16))) <= P
    pools = [workloads.device_layer_pool(1000 + l, P, dev()) for l in range(LAYERS)]
    rng = np.random.Generator(np.random.PCG64(44))
    qs = [to_dev(rng.standard_normal((B, 40, 128), dtype=np.float32).astype(np.float16))
          for _ in range(LAYERS)]
    kn = [to_dev(rng.standard_normal((B, 10, 128), dtype=np.float32).astype(np.float16))
          for _ in range(LAYERS)]
    vn = [to_dev(rng.standard_normal((B, 10, 128), dtype=np.float32).astype(np.float16))
          for _ in range(LAYERS)]
    L = lay.seq_lens.astype(np.int64)
    slots = (lay.block_table[np.arange(B), (L - 1) // 16].astype(np.int64) * 16 + (L - 1) % 16)
    # host copies of the checked layers' pools, taken before any kernel runs;
    # the oracle appends each sequence's new token, then attends over every
    # sequence of the batch
    ref = {}
    bt = np.ascontiguousarray(lay.block_table, np.int32)
    for l in CHECKED_LAYERS:
        okc = pools[l][0].cpu().numpy()
        ovc = pools[l][1].cpu().numpy()
        vs = pools[l][2].cpu().numpy()
        oracle.kv_append(kn[l].cpu().numpy(), vn[l].cpu().numpy(), slots, vs, okc, ovc)
        r = oracle.paged_decode(qs[l].cpu().numpy(), okc, ovc, vs, bt, lay.seq_lens,
                                workloads.default_sm_scale(128))
        ref[l] = (r["out"], r["lse"])
        del okc, ovc
    step = MultiLayerDecode([p[0] for p in pools], [p[1] for p in pools], [p[2] for p in pools],
                            to_dev(lay.block_table), to_dev(lay.seq_lens), to_dev(slots),
                            int(L.max()), 40, split_chunk=512)
    outs = [torch.empty((B, 40, 128), dtype=torch.float16, device=dev()) for _ in range(LAYERS)]
    lses = [torch.empty((B, 40), dtype=torch.float32, device=dev()) for _ in range(LAYERS)]
    return dict(K=K, lay=lay, pools=pools, qs=qs, kn=kn, vn=vn, slots=slots, ref=ref,
                step=step, outs=outs, lses=lses)


def check_layers(s, outs, lses):
    """Every sequence of the checked layers against the oracle."""
    for l in CHECKED_LAYERS:
        ro, rl = s["ref"][l]
        check_close(outs[l].float().cpu().numpy(), ro, lses[l].cpu().numpy(), rl)


def test_fullpool_eager_step_matches_oracle(setup):
    s = setup
    s["step"].step(s["qs"], s["kn"], s["vn"], s["outs"], s["lses"])
    assert s["step"].check() == 0
    check_layers(s, s["outs"], s["lses"])


def test_fullpool_graph_replay_matches_eager(setup):
    s = setup
    ref = [o.clone() for o in s["outs"]]
    ref_l = [x.clone() for x in s["lses"]]
    for o in s["outs"]:
        o.fill_(float("nan"))
    s["step"].capture(s["qs"], s["kn"], s["vn"], s["outs"], s["lses"])
    for o in s["outs"]:
        o.fill_(float("nan"))
    s["step"].replay()
    assert s["step"].check() == 0
    for l in range(LAYERS):
        assert torch.equal(s["outs"][l], ref[l]) and torch.equal(s["lses"][l], ref_l[l])


def test_scale_validation_rejects_bad_scale(setup):
    from fp8_paged_kv_append_gb300.decode_step import ScaleError, validate_scales
    bad = [p[2].clone() for p in setup["pools"][:2]]
    bad[1][3] = float("nan")
    with pytest.raises(ScaleError):
        validate_scales(bad)
    bad[1][3] = 0.0
    with pytest.raises(ScaleError):
        validate_scales(bad)


@pytest.mark.parametrize("schedule", ["balanced", "balanced_fused", "fused", "whole", "auto"])
def test_fullpool_other_schedules_match_oracle(setup, schedule):
    """The same 40-layer step on the load-balanced split (block table and
    lengths read ahead of the wait on the preceding kernel), with and without
    the append folded in, the chunked split with the append folded in, one
    CTA per (sequence, KV head) writing the output itself (one launch per
    layer), and the automatic choice (captured graph each): every sequence of layers 0,
    17 and 39 against the oracle.  Folded-in appends write the same bytes to the
    same slots as the separate append."""
    from fp8_paged_kv_append_gb300.decode_step import MultiLayerDecode
    s = setup
    lay, B = s["lay"], len(s["lay"].seq_lens)
    step = MultiLayerDecode([p[0] for p in s["pools"]], [p[1] for p in s["pools"]],
                            [p[2] for p in s["pools"]], to_dev(lay.block_table),
                            to_dev(lay.seq_lens), to_dev(s["slots"]),
                            int(lay.seq_lens.max()), 40, schedule=schedule)
    if schedule == "auto":
        assert step.schedule == "fused"  # 225 tiles per CTA on 152 SMs
    outs = [torch.full((B, 40, 128), float("nan"), dtype=torch.float16, device=dev())
            for _ in range(LAYERS)]
    lses = [torch.full((B, 40), float("nan"), dtype=torch.float32, device=dev())
            for _ in range(LAYERS)]
    step.capture(s["qs"], s["kn"], s["vn"], outs, lses)
    for o in outs:
        o.fill_(float("nan"))
    step.replay()
    assert step.check() == 0
    check_layers(s, outs, lses)
    for l in range(LAYERS):  # every row of every layer written (no NaN left from the fill)
        assert not torch.isnan(outs[l]).any() and not torch.isnan(lses[l]).any()
