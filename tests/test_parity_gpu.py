"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle on
the same seeded inputs.  Every case compares every output element, the five
full-size workloads (and the head-dim-256 one) included; cases with more work
items than CTAs run the persistent kernels' item-to-item carry-over."""
import math

import numpy as np
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from parity import check, run_and_check, run_gpu, run_oracle, to_dev
from tiled_online_softmax_02_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_02_gb300 import build
    build.build()
    attn.load_library()
    torch.cuda.set_device(0)


# --- the five workloads, scaled so the oracle runs in seconds; every case
# --- spans several key / query tiles and ends in a ragged tail
SMALL = {
    "tiny_f32": WORKLOADS["tiny_f32"],
    "dit_f32": WORKLOADS["dit_f32"].replace(Hq=3, Hkv=3, Sq=300, Sk=300, kv_capacity=300),
    "gqa_causal_bf16": WORKLOADS["gqa_causal_bf16"].replace(Hq=4, Hkv=2, Sq=600, Sk=600,
                                                            kv_capacity=600),
    "window_softcap_bf16": WORKLOADS["window_softcap_bf16"].replace(
        B=2, Hq=4, Hkv=2, Sq=1000, Sk=1000, kv_capacity=1000, local_window=256),
    "ragged_kvcache_f16": WORKLOADS["ragged_kvcache_f16"].replace(
        B=3, Hq=8, Hkv=2, Sq=100, Sk=700, kv_capacity=700),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_small(name):
    run_and_check(SMALL[name])


# --- feature matrix per dtype and head dim
def _base(dtype, D, **kw):
    w = Workload("case", B=2, Hq=4, Hkv=2, Sq=200, Sk=200, kv_capacity=200, D=D, dtype=dtype,
                 causal=False, seed=1234)
    return w.replace(**kw)


FEATURES = {
    "noncausal": {},
    "causal": {"causal": True},
    "causal_sq_lt_sk": {"causal": True, "Sq": 70, "Sk": 333, "kv_capacity": 333},
    "sq_gt_sk_causal": {"causal": True, "Sq": 300, "Sk": 150, "kv_capacity": 150},
    "window_causal": {"causal": True, "local_window": 130},
    "window_noncausal": {"local_window": 77},
    "softcap_1": {"softcap": 1.0, "q_std": 2.0, "k_std": 2.0},
    "softcap_50_causal": {"softcap": 50.0, "causal": True},
    "mask_per_head": {"mask": "per_head", "mask_neg_inf_frac": 0.2},
    "mask_shared_causal": {"mask": "shared", "mask_neg_inf_frac": 0.1, "causal": True},
    "mask_sk_not_mult4": {"mask": "per_batch", "Sk": 203, "kv_capacity": 203, "causal": True},
    "token_major": {"out_layout": 1, "causal": True},
    "gqa_group4": {"Hq": 8, "Hkv": 2, "causal": True},
    "mha": {"Hq": 3, "Hkv": 3},
    "ragged_finite_garbage": {"ragged": True, "Sq": 50, "Sk": 400, "kv_capacity": 400,
                              "causal": True, "garbage": "finite"},
    "ragged_nonfinite_garbage": {"ragged": True, "Sq": 50, "Sk": 400, "kv_capacity": 400,
                                 "causal": True, "garbage": "nonfinite"},
    "sk_lt_capacity_garbage": {"Sk": 180, "kv_capacity": 260, "garbage": "nonfinite"},
    "everything": {"ragged": True, "Sq": 64, "Sk": 512, "kv_capacity": 512, "causal": True,
                   "local_window": 200, "softcap": 5.0, "mask": "per_head",
                   "mask_neg_inf_frac": 0.1, "garbage": "nonfinite", "out_layout": 1},
    "negative_scale": {"scale": -0.05},
    "large_scores": {"q_std": 4.0, "k_std": 4.0, "causal": True},
}

DTYPE_D = [("f32", 64), ("f32", 128), ("f32", 40), ("f32", 96), ("f32", 200), ("f32", 256),
           ("f32", 330), ("f32", 384), ("bf16", 64), ("bf16", 128), ("f16", 64), ("f16", 128),
           ("bf16", 256), ("f16", 256), ("bf16", 384), ("f16", 384)]


@pytest.mark.parametrize("feature", list(FEATURES))
@pytest.mark.parametrize("dtype,D", DTYPE_D, ids=[f"{a}-d{b}" for a, b in DTYPE_D])
def test_feature(dtype, D, feature):
    run_and_check(_base(dtype, D, **FEATURES[feature]), what=f"{feature} {dtype} D={D}")


# --- edge cases
EDGES = {
    "sq1_decode": {"Sq": 1, "Sk": 517, "kv_capacity": 517, "causal": True},
    "sk1": {"Sq": 33, "Sk": 1, "kv_capacity": 1},
    "sq1_sk1": {"Sq": 1, "Sk": 1, "kv_capacity": 1, "causal": True},
    "exact_tiles": {"Sq": 256, "Sk": 256, "kv_capacity": 256, "causal": True},
    "one_past_tile": {"Sq": 129, "Sk": 129, "kv_capacity": 129, "causal": True},
    "rows_without_keys": {"Sq": 300, "Sk": 100, "kv_capacity": 100, "causal": True},
    "window1": {"causal": True, "local_window": 1},
    "all_masked_rows": {"mask": "per_batch", "mask_neg_inf_frac": 1.0},
    "mostly_masked": {"mask": "per_batch", "mask_neg_inf_frac": 0.97, "causal": True},
}


EDGE_DTYPE_D = [("f32", 64), ("f32", 384), ("bf16", 128), ("f16", 64), ("bf16", 256), ("f16", 384)]


@pytest.mark.parametrize("edge", list(EDGES))
@pytest.mark.parametrize("dtype,D", EDGE_DTYPE_D, ids=[f"{a}-d{b}" for a, b in EDGE_DTYPE_D])
def test_edge(dtype, D, edge):
    run_and_check(_base(dtype, D, **EDGES[edge]), what=f"{edge} {dtype} D={D}")


@pytest.mark.parametrize("dtype,D", [("f32", 64), ("bf16", 128), ("f16", 64)])
def test_inconsistent_lengths(dtype, D):
    """total != past + Sq, total beyond Sk, negative past: the per-row rule
    still decides (rows whose causal limit is below 0 are zero)."""
    w = _base(dtype, D, Sq=40, Sk=300, kv_capacity=320, causal=True, garbage="nonfinite")
    x = make_inputs(w)
    x["total_lengths"] = torch.tensor([500, 120], dtype=torch.int32)
    x["past_lengths"] = torch.tensor([-10, 30], dtype=torch.int32)
    # garbage only beyond what any row may see: slots >= min(total, Sk)
    for b, lim in enumerate([300, 120]):
        x["k"][b, :, lim:] = float("nan")
        x["v"][b, :, lim:] = float("inf")
    out = run_gpu(w, x)
    check(w, out.double().cpu().numpy(), run_oracle(w, x), f"inconsistent lengths {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sk_zero_writes_zeros(dtype):
    w = _base(dtype, 64, Sk=0, kv_capacity=16)
    x = make_inputs(w)
    g = to_dev(x)
    out = torch.full((w.B, w.Hq, w.Sq, w.D), 7.0, dtype=g["q"].dtype, device="cuda")
    attn.attn_fwd(g["q"], g["k"], g["v"], seq_k=0, out=out)
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_empty_batch_is_noop():
    q = torch.zeros(0, 2, 8, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(0, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    out = attn.attn_fwd(q, k, k)
    assert out.shape == (0, 2, 8, 64)


def test_head_dim_256_long_rows():
    """D = 256 (single-lane kernel): several query tiles, dozens of key tiles,
    GQA, causal with ragged tails; and the ragged cache with non-finite garbage."""
    run_and_check(_base("bf16", 256, Hq=8, Hkv=2, Sq=700, Sk=1400, kv_capacity=1500, causal=True))
    run_and_check(_base("f16", 256, ragged=True, Sq=90, Sk=900, kv_capacity=900, causal=True,
                        garbage="nonfinite", mask="per_batch", mask_neg_inf_frac=0.1))


def test_head_dim_384_long_rows():
    """D = 384 (single-lane kernel, Q in shared memory, 32-key tiles): many key
    tiles, GQA, causal with ragged tails; the ragged cache with non-finite
    garbage and a mask; soft-cap with a window; the fp32 CUDA-core kernel."""
    run_and_check(_base("bf16", 384, Hq=8, Hkv=2, Sq=700, Sk=1400, kv_capacity=1500, causal=True))
    run_and_check(_base("f16", 384, ragged=True, Sq=90, Sk=900, kv_capacity=900, causal=True,
                        garbage="nonfinite", mask="per_batch", mask_neg_inf_frac=0.1))
    run_and_check(_base("bf16", 384, Sq=333, Sk=700, kv_capacity=700, causal=True, local_window=150,
                        softcap=10.0, out_layout=1))
    run_and_check(_base("f32", 384, Hq=8, Hkv=2, Sq=300, Sk=700, kv_capacity=700, causal=True,
                        mask="per_head", mask_neg_inf_frac=0.1))


@pytest.mark.parametrize("D", [256, 384])
def test_wide_head_dim_splitkv_unsupported(D):
    q = torch.zeros(1, 2, 8, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_splitkv(q, q, q, num_splits=2)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED


def test_unsupported_head_dim_raises():
    q = torch.zeros(1, 1, 8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd(q, q, q)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED


# --- the page's f16 regression protocol, with our own generator
def test_f16_prefill_protocol():
    """B=1, Hq=14, Hkv=2, D=64, causal, Sq=Sk=kv_capacity over a sweep of
    lengths and input amplitudes 1 and 3; gates: all finite, max abs error
    < 2e-3 at amplitude 1, max relative error (denominator floored at 1e-2)
    < 6e-3 at every amplitude.

    Values are uniform on [-amp, 0): that is the range the page's generator
    actually produces (a 31-bit state divided by 2^32 - 1 lies in [0, 0.5),
    so 2u - 1 lies in [-1, 0)), and the gates were set on such data, whose
    outputs stay away from 0.  Symmetric data puts outputs near 0, where the
    1e-2 floor turns the 16-bit rounding of P (which the page's kernel does
    too) into large relative numbers; the general tolerance tests cover it."""
    worst_abs, worst_rel = 0.0, 0.0
    rng = np.random.default_rng(0x9E3779B9)
    for amp in (1.0, 3.0):
        for seq in (2, 4, 8, 16, 30, 64, 96, 128, 192, 256, 300):
            w = Workload("f16_protocol", B=1, Hq=14, Hkv=2, Sq=seq, Sk=seq, kv_capacity=seq, D=64,
                         dtype="f16", causal=True)
            x = {"q": torch.from_numpy(rng.uniform(-amp, 0.0, (1, 14, seq, 64)).astype(np.float32)).half(),
                 "k": torch.from_numpy(rng.uniform(-amp, 0.0, (1, 2, seq, 64)).astype(np.float32)).half(),
                 "v": torch.from_numpy(rng.uniform(-amp, 0.0, (1, 2, seq, 64)).astype(np.float32)).half(),
                 "mask": None, "total_lengths": None, "past_lengths": None}
            got = run_gpu(w, x).double().cpu().numpy()
            ref = run_oracle(w, x)
            assert np.isfinite(got).all()
            err = np.abs(got - ref)
            worst_rel = max(worst_rel, float((err / np.maximum(np.abs(ref), 1e-2)).max()))
            if amp == 1.0:
                worst_abs = max(worst_abs, float(err.max()))
    assert worst_abs < 2e-3, worst_abs
    assert worst_rel < 6e-3, worst_rel


@pytest.mark.parametrize("amp", [1.0, 3.0])
def test_f16_prefill_symmetric_data(amp):
    """The same sweep on symmetric data, held to the general 16-bit tolerance."""
    rng = np.random.default_rng(77)
    for seq in (2, 30, 128, 300):
        w = Workload("f16_sym", B=1, Hq=14, Hkv=2, Sq=seq, Sk=seq, kv_capacity=seq, D=64,
                     dtype="f16", causal=True)
        x = {"q": torch.from_numpy(rng.uniform(-amp, amp, (1, 14, seq, 64)).astype(np.float32)).half(),
             "k": torch.from_numpy(rng.uniform(-amp, amp, (1, 2, seq, 64)).astype(np.float32)).half(),
             "v": torch.from_numpy(rng.uniform(-amp, amp, (1, 2, seq, 64)).astype(np.float32)).half(),
             "mask": None, "total_lengths": None, "past_lengths": None}
        check(w, run_gpu(w, x).double().cpu().numpy(), run_oracle(w, x), f"f16 symmetric {seq}")


# --- invariances of the CUDA path itself
@pytest.mark.parametrize("dtype,D", [("f32", 128), ("bf16", 128), ("f16", 64)])
def test_garbage_slots_do_not_change_output(dtype, D):
    w = _base(dtype, D, ragged=True, Sq=60, Sk=500, kv_capacity=500, causal=True,
              mask="per_batch", mask_neg_inf_frac=0.1, garbage="finite")
    a = make_inputs(w)
    b = dict(a, k=a["k"].clone(), v=a["v"].clone())
    for i, t in enumerate(a["total_lengths"].tolist()):  # only slots >= total change
        b["k"][i, :, t:] = float("nan")
        b["v"][i, :, t:] = float("-inf") if i % 2 else float("inf")
    oa = run_gpu(w, a)
    ob = run_gpu(w, b)
    assert torch.equal(oa, ob)


def test_deterministic():
    w = SMALL["gqa_causal_bf16"]
    x = make_inputs(w)
    assert torch.equal(run_gpu(w, x), run_gpu(w, x))


def test_host_tensors_end_to_end():
    """CPU (pinned) inputs go through the same kernels and come back on the host."""
    w = SMALL["ragged_kvcache_f16"]
    x = make_inputs(w)
    dev_out = run_gpu(w, x).cpu()
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    host_out = attn.attn_fwd(pin["q"], pin["k"], pin["v"], mask=pin["mask"],
                             total_lengths=pin["total_lengths"], past_lengths=pin["past_lengths"],
                             causal=w.causal, scale=w.softmax_scale, seq_k=w.Sk)
    assert not host_out.is_cuda
    assert torch.equal(host_out, dev_out)


# --- failure detection: a bounded wait that runs out reports, and the
# --- context stays usable
def test_bounded_wait_times_out_and_reports():
    assert attn.get_device_status() == attn.ATTN_OK
    st = attn.selftest_bounded_wait(2_000_000)  # 2 ms on a barrier nobody arrives at
    assert st == attn.ATTN_ERR_TIMEOUT
    assert attn.get_device_status() == attn.ATTN_OK  # the query cleared it
    run_and_check(SMALL["tiny_f32"])  # the context still works


# --- more work items than the persistent kernels have CTAs (one per SM): a
# --- CTA runs several items in turn, so the K/V ring, the barrier phases, the
# --- snake order, the cost-ranked batches and tensor memory carry over from
# --- item to item -- here under a check of every output element
MULTI_ITEM = {
    # tile kernel, two query tiles per item: 2 * 48 * ceil(400 / 256) = 192 items
    # (single-lane kernels: 2 * 48 * ceil(400 / 128) = 384)
    "two_tile_causal": dict(B=2, Hq=48, Hkv=8, Sq=400, Sk=400, kv_capacity=400, causal=True),
    # key-split lanes (Sq <= 128): 4 * 48 = 192 items, ragged lengths ranked by
    # cost, a per-batch mask (staged asynchronously at D = 128), NaN / Inf
    # garbage past each valid length
    "keysplit_ragged_mask": dict(B=4, Hq=48, Hkv=8, Sq=100, Sk=900, kv_capacity=900, causal=True,
                                 ragged=True, mask="per_batch", mask_neg_inf_frac=0.1,
                                 garbage="nonfinite"),
    # both item kinds in one launch (the last query pair holds one tile):
    # 2 * 40 * 3 = 240 items, window and soft-cap, token-major output
    "mixed_window_softcap": dict(B=2, Hq=40, Hkv=8, Sq=520, Sk=520, kv_capacity=520, causal=True,
                                 local_window=200, softcap=20.0, out_layout=1),
}
MULTI_DTYPE_D = [("bf16", 64), ("bf16", 128), ("f16", 64), ("f16", 128), ("bf16", 256),
                 ("f16", 256), ("bf16", 384), ("f16", 384), ("f32", 128), ("f32", 384)]


@pytest.mark.parametrize("case", list(MULTI_ITEM))
@pytest.mark.parametrize("dtype,D", MULTI_DTYPE_D, ids=[f"{a}-d{b}" for a, b in MULTI_DTYPE_D])
def test_more_items_than_ctas(dtype, D, case):
    run_and_check(_base(dtype, D, **MULTI_ITEM[case]), what=f"multi-item {case} {dtype} D={D}")


# --- full-size workloads: every output element against the oracle (the
# --- oracle's threaded fp64 path; the largest take seconds on the host)
FULL_SIZE = dict(WORKLOADS, **{n: EXTRA_WORKLOADS[n] for n in
                                ("gqa_causal_bf16_d256", "gqa_causal_bf16_d384", "vae_f32_d384")})


@pytest.mark.parametrize("name", list(FULL_SIZE))
def test_workload_full_size_every_row(name):
    w = FULL_SIZE[name]
    x = make_inputs(w)
    out = run_gpu(w, x)
    got = out.double().cpu().numpy()
    del out
    check(w, got, run_oracle(w, x), f"{name} full size, every row")
