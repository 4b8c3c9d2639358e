"""The seeded input generators: shapes, dtypes, determinism, lengths and
garbage placement, and the row sampler (CPU only)."""
import numpy as np
import pytest
import torch

from tiled_online_softmax_02_gb300.inputs import WORKLOADS, make_inputs, sample_rows


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_sample_rows_terminates_and_is_valid(name):
    w = WORKLOADS[name]
    for n in (1, 160, 10_000):
        rows = sample_rows(w, n)
        assert 0 < len(rows) <= min(max(n, 1), w.B * w.Hq * w.Sq) or len(rows) <= n + 64
        assert len({tuple(r) for r in rows}) == len(rows)
        assert (rows[:, 0] >= 0).all() and (rows[:, 0] < w.B).all()
        assert (rows[:, 1] >= 0).all() and (rows[:, 1] < w.Hq).all()
        assert (rows[:, 2] >= 0).all() and (rows[:, 2] < w.Sq).all()


def test_small_inputs_deterministic_and_shaped():
    w = WORKLOADS["ragged_kvcache_f16"].replace(B=3, Hq=8, Hkv=2, Sq=20, Sk=300, kv_capacity=320)
    a, b = make_inputs(w), make_inputs(w)
    for k in ("q", "k", "v", "mask", "total_lengths", "past_lengths"):
        assert torch.equal(a[k], b[k])
    assert a["q"].shape == (3, 8, 20, 128) and a["q"].dtype == torch.float16
    assert a["k"].shape == (3, 2, 320, 128)
    assert a["mask"].shape == (3, 20, 300) and a["mask"].dtype == torch.float32
    assert torch.equal(a["total_lengths"], a["past_lengths"] + 20)
    assert int(a["past_lengths"].max()) <= 300 - 20
    frac = float(torch.isneginf(a["mask"]).float().mean())
    assert 0.05 < frac < 0.15
    for i, t in enumerate(a["total_lengths"].tolist()):
        assert float(a["v"][i, :, t:].abs().float().min()) >= 0  # garbage is finite
        assert torch.isfinite(a["v"][i, :, t:].float()).all()


def test_workload_table_matches_the_five_configs():
    w = WORKLOADS
    assert (w["tiny_f32"].B, w["tiny_f32"].Hq, w["tiny_f32"].Hkv, w["tiny_f32"].Sq, w["tiny_f32"].D) == (1, 2, 1, 64, 64)
    assert w["dit_f32"].out_layout == 1 and not w["dit_f32"].causal and w["dit_f32"].Hq == 24
    assert (w["gqa_causal_bf16"].B, w["gqa_causal_bf16"].Hq, w["gqa_causal_bf16"].Hkv,
            w["gqa_causal_bf16"].Sq) == (2, 32, 8, 4096)
    c4 = w["window_softcap_bf16"]
    assert (c4.local_window, c4.softcap, round(c4.q_std ** 2, 6)) == (1024, 50.0, 2.0)
    c5 = w["ragged_kvcache_f16"]
    assert (c5.B, c5.Hq, c5.Hkv, c5.Sq, c5.kv_capacity, c5.mask_planes) == (8, 32, 4, 128, 4096, 8)
    assert [x.seed for x in w.values()] == [0xA77E0000 + i for i in range(5)]
