"""Split-KV attention (attn_fwd_splitkv): the output and the row log-sum-exp
against the fp64 oracle on the same seeded inputs, for several split counts,
decode-shaped problems and the masking features."""
import numpy as np
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from parity import check, check_lse, lse_tolerance, run_gpu, run_gpu_splitkv, run_oracle_lse
from tiled_online_softmax_02_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_02_gb300 import build
    build.build()
    attn.load_library()
    torch.cuda.set_device(0)


def _w(dtype="bf16", D=128, **kw):
    w = Workload("splitkv", B=2, Hq=8, Hkv=2, Sq=1, Sk=1500, kv_capacity=1500, D=D, dtype=dtype,
                 causal=True, seed=4321)
    return w.replace(**kw)


CASES = {
    "decode": {},
    "decode_ragged": {"ragged": True, "Sk": 2000, "kv_capacity": 2048, "garbage": "nonfinite"},
    "decode_noncausal_d64": {"causal": False, "D": 64},
    "chunk_prefill_mask": {"Sq": 100, "ragged": True, "Sk": 1200, "kv_capacity": 1200,
                           "mask": "per_batch", "mask_neg_inf_frac": 0.1, "garbage": "finite"},
    "prefill_two_query_tiles": {"Sq": 300, "Sk": 900, "kv_capacity": 900},
    "window_softcap": {"Sq": 260, "Sk": 1400, "kv_capacity": 1400, "local_window": 300,
                       "softcap": 20.0},
    "token_major_f16": {"dtype": "f16", "Sq": 40, "Sk": 777, "kv_capacity": 800, "out_layout": 1},
    "mask_per_head_window": {"Sq": 3, "Sk": 640, "kv_capacity": 640, "mask": "per_head",
                             "mask_neg_inf_frac": 0.3, "local_window": 200},
}


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 0])
@pytest.mark.parametrize("case", list(CASES))
def test_splitkv_matches_oracle(case, splits):
    w = _w(**CASES[case])
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, splits)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, f"{case} splits={splits}")
    check_lse(lse.cpu().numpy(), ref_lse, f"{case} splits={splits} lse", tol=lse_tolerance(w, x))


def test_more_splits_than_key_tiles():
    w = _w(Sk=200, kv_capacity=256)  # two key tiles, up to 64 splits
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, 64)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, "64 splits over 2 tiles")
    check_lse(lse.cpu().numpy(), ref_lse, "64 splits lse", tol=lse_tolerance(w, x))


def test_rows_without_keys_have_lse_minus_inf():
    w = _w(Sq=40, Sk=20, kv_capacity=20)  # causal with Sq > Sk: rows 0..19 see nothing
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, 2)
    ref, ref_lse = run_oracle_lse(w, x)
    assert np.isneginf(ref_lse[:, :, :20]).all()
    check(w, out.double().cpu().numpy(), ref, "rows without keys")
    check_lse(lse.cpu().numpy(), ref_lse, "rows without keys lse", tol=lse_tolerance(w, x))


def test_one_split_equals_attn_fwd():
    w = _w(Sq=130, Sk=700, kv_capacity=700, ragged=True)
    x = make_inputs(w)
    out, _ = run_gpu_splitkv(w, x, 1)
    assert torch.equal(out, run_gpu(w, x))


def test_sk_zero():
    w = _w(Sk=0, kv_capacity=16)
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, 4)
    assert bool((out == 0).all()) and bool(torch.isneginf(lse).all())


def test_f32_is_unsupported():
    q = torch.zeros(1, 1, 4, 64, device="cuda")
    with pytest.raises(ValueError):
        attn.attn_fwd_splitkv(q, q, q)


def test_ragged_kvcache_full_size_auto_splits():
    """The full ragged KV-cache workload through the split path: every output
    element and every row log-sum-exp."""
    w = WORKLOADS["ragged_kvcache_f16"]
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, 0)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, "ragged kv-cache split-KV, every row")
    check_lse(lse.cpu().numpy(), ref_lse, "ragged kv-cache split-KV lse", tol=lse_tolerance(w, x))


# more (query pair, split range) items than CTAs: each persistent CTA takes
# several, so its rings and barrier phases carry across items and split ranges
MULTI_ITEM = {
    "two_tile_items": dict(B=2, Hq=40, Hkv=8, Sq=300, Sk=1200, kv_capacity=1200, causal=True),
    "keysplit_items_mask": dict(B=4, Hq=48, Hkv=8, Sq=100, Sk=1000, kv_capacity=1024, ragged=True,
                                mask="per_batch", mask_neg_inf_frac=0.1, garbage="nonfinite"),
}


@pytest.mark.parametrize("splits", [2, 3])
@pytest.mark.parametrize("case", list(MULTI_ITEM))
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64)])
def test_more_items_than_ctas(dtype, D, case, splits):
    w = _w(dtype, D, **MULTI_ITEM[case])
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, splits)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, f"multi-item {case} splits={splits}")
    check_lse(lse.cpu().numpy(), ref_lse, f"multi-item {case} splits={splits} lse",
              tol=lse_tolerance(w, x))
