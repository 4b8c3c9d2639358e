"""The bench's host-side bookkeeping on CPU: the attention FLOP count against
the oracle's own visible keys, the DSA workloads' FLOP and byte counts against
hand counts, both reference arms (the CPU oracle timed on a bounded sample)
printing a well-formed JSON line, and the ncu traffic table belonging to the
kernel sources in the tree."""
import contextlib
import io
import json

import numpy as np
import pytest

import bench
from tiled_online_softmax_02_gb300.inputs import DsaWorkload, make_dsa_inputs


def test_dsa_allowed_counts_and_flops():
    w = DsaWorkload("t", B=2, S=3, H=5, D=8, T=10, top_k=4, dtype="bf16", bias="causal")
    x = make_dsa_inputs(w)
    cnt = bench.dsa_allowed_counts(x)
    # causal: row s allows keys t <= T - S + s
    exp = np.array([[w.T - w.S + s + 1 for s in range(w.S)]] * w.B)
    assert np.array_equal(cnt, exp)
    assert bench.dsa_flops(w, cnt) == 2 * w.H * w.D * int(exp.sum())


def test_dsa_algorithmic_bytes():
    w = DsaWorkload("t", B=2, S=3, H=5, D=8, T=10, top_k=4, dtype="bf16")
    rows = 6
    exp = (rows * 5 * 8 * 2 + 2 * 10 * 8 * 2 + rows * 5 * 2  # query, key, weights
           + rows * 10 * 4 + 2 * rows * 10 * 4 + rows * 4 * 8)  # bias, scores twice, indices
    assert bench.dsa_algorithmic_bytes(w) == exp
    assert bench.dsa_algorithmic_bytes(w.replace(dtype="f32")) == exp + rows * 5 * 8 * 2 + 2 * 10 * 8 * 2 + rows * 5 * 2


def _reference_line(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(argv) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["dsa_decode_bf16", "tiny_f32"])
def test_reference_arm_prints_one_line(workload):
    d = _reference_line(["--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "3",
                         "--ref-seconds", "2"])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == workload
    assert d["steps"] == 1 and d["warmup"] == 3


VISIBILITY_CASES = {
    "causal_square": dict(B=2, Hq=2, Hkv=1, Sq=40, Sk=40, kv_capacity=40, causal=True),
    "causal_sq_gt_sk": dict(B=1, Hq=2, Hkv=2, Sq=50, Sk=30, kv_capacity=30, causal=True),
    "window_no_causal": dict(B=2, Hq=2, Hkv=1, Sq=24, Sk=64, kv_capacity=64, causal=False, local_window=9),
    "window_causal": dict(B=1, Hq=4, Hkv=2, Sq=33, Sk=70, kv_capacity=72, causal=True, local_window=17),
    "ragged_cache": dict(B=3, Hq=2, Hkv=1, Sq=16, Sk=90, kv_capacity=96, causal=True, ragged=True),
    "explicit_lengths": dict(B=3, Hq=2, Hkv=2, Sq=20, Sk=48, kv_capacity=64, causal=True,
                             total=[70, 30, 5], past=[40, 25, 0]),
    "masked_per_head": dict(B=2, Hq=2, Hkv=1, Sq=12, Sk=36, kv_capacity=36, causal=True, mask="per_head",
                            mask_neg_inf_frac=0.3),
}


@pytest.mark.parametrize("case", list(VISIBILITY_CASES))
def test_flop_count_matches_the_oracles_visible_keys(case):
    """The bench's FLOP count rests on visible_counts (keys a row sees under
    the length, causal and window limits) and on the -inf mask entries among
    them.  Both are checked against the oracle itself: with Q = K = 0 every
    visible key of a row gets the same weight, and with V's rows one-hot per
    key slot the oracle's output row is 1 / count on exactly the keys the
    row sees (a 0 / -inf mask removes the -inf keys and leaves the rest
    uniform)."""
    import oracle
    import torch
    from tiled_online_softmax_02_gb300.inputs import Workload, make_inputs
    kw = dict(VISIBILITY_CASES[case])
    total, past = kw.pop("total", None), kw.pop("past", None)
    w = Workload("vis", dtype="f32", seed=77, D=kw["kv_capacity"], **kw)
    x = make_inputs(w)
    if total is not None:
        x["total_lengths"] = torch.tensor(total, dtype=torch.int32)
        x["past_lengths"] = torch.tensor(past, dtype=torch.int32)
    if x["mask"] is not None:  # keep the -inf entries, zero the rest: weights stay uniform
        x["mask"] = torch.where(torch.isneginf(x["mask"]), x["mask"], torch.zeros_like(x["mask"]))
    C = w.kv_capacity
    q = np.zeros((w.B, w.Hq, w.Sq, C), np.float32)
    k = np.zeros((w.B, w.Hkv, C, C), np.float32)
    v = np.broadcast_to(np.eye(C, dtype=np.float32), (w.B, w.Hkv, C, C)).copy()
    out = oracle.attn_fwd(q, k, v, B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk, kv_capacity=C, D=C,
                          causal=w.causal, local_window=w.local_window, mask=x["mask"],
                          mask_planes=w.mask_planes, total_lengths=x["total_lengths"],
                          past_lengths=x["past_lengths"])
    seen = out > 0  # [B, Hq, Sq, C]: the keys each row's output draws on
    cnt = seen.sum(axis=-1)
    # uniform weights over the keys seen, as the construction promises
    assert np.allclose(out.sum(axis=-1)[cnt > 0], 1.0)
    assert np.allclose(out[seen], np.broadcast_to(1.0 / np.maximum(cnt, 1)[..., None], out.shape)[seen])
    tot = x["total_lengths"].numpy() if x["total_lengths"] is not None else None
    pst = x["past_lengths"].numpy() if x["past_lengths"] is not None else None
    vis = bench.visible_counts(w, tot, pst)  # [B, Sq], the same for every head
    flops, excl = bench.flops_of(w, x)
    if x["mask"] is None:
        assert np.array_equal(cnt, np.broadcast_to(vis[:, None, :], cnt.shape))
        assert flops == excl == 4 * w.D * int(cnt.sum())
    else:
        assert np.all(cnt <= vis[:, None, :])
        assert flops == 4 * w.D * w.Hq * int(vis.sum())
        assert excl == 4 * w.D * int(cnt.sum())
        assert excl < flops  # the case masks some visible keys


def test_traffic_table_belongs_to_the_committed_sources():
    """Every DRAM-traffic figure the bench reports was captured on the
    kernel sources in the tree: its entry's source hash is that kernel
    family's current hash (a kernel change without a new capture reports
    traffic null, which this catches before a run does)."""
    for key, ent in bench.NCU_TRAFFIC.items():
        name, *flags = key.split("+")
        if name in bench.DSA_WORKLOADS:
            family = "dsa"
        else:
            w = bench.ALL_WORKLOADS[name]
            family = bench.kernel_family(w, "splitkv" in flags, "f32split" in flags)
        assert ent["bytes_per_launch"] > 0
        assert ent["source_hash"] == bench.kernel_source_hash(family), key
