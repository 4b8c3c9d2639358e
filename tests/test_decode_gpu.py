"""The few-rows (decode) kernel: problems with (Hq / Hkv) * Sq <= 32 query rows
per kv head, through attn_fwd and attn_fwd_splitkv, against the fp64 oracle
on the same seeded inputs -- every row count around the 16 / 32 variants,
both head dims and 16-bit types, causal rows with different limits, window,
soft-cap, the three mask broadcasts, token-major output, NaN / Inf garbage
past the valid length, rows without keys, a running maximum that keeps
growing, and every row of the full-size decode workload."""
import numpy as np
import pytest
import torch

from parity import (check, check_lse, lse_tolerance, run_gpu, run_gpu_splitkv, run_oracle,
                    run_oracle_lse)
from tiled_online_softmax_02_gb300.inputs import EXTRA_WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tiled_online_softmax_02_gb300 as attn
    from tiled_online_softmax_02_gb300 import build
    build.build()
    attn.load_library()
    torch.cuda.set_device(0)


def _w(dtype="bf16", D=128, **kw):
    w = Workload("decode", B=3, Hq=8, Hkv=2, Sq=1, Sk=1000, kv_capacity=1024, D=D, dtype=dtype,
                 causal=True, ragged=True, garbage="finite", seed=777)
    return w.replace(**kw)


# (Hq, Hkv, Sq): query rows per kv head = Hq / Hkv * Sq
ROW_SHAPES = {
    "rows1_mha": (4, 4, 1),
    "rows2": (4, 2, 1),
    "rows15": (15, 1, 1),
    "rows16_gqa": (32, 2, 1),
    "rows16_sq4": (8, 2, 4),
    "rows17": (17, 1, 1),
    "rows24_sq3": (16, 2, 3),
    "rows32_sq2": (32, 2, 2),
    "rows32_sq32": (2, 2, 32),
}


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("bf16", 64), ("f16", 128)])
@pytest.mark.parametrize("shape", list(ROW_SHAPES))
def test_row_counts_attn_fwd(shape, dtype, D):
    Hq, Hkv, Sq = ROW_SHAPES[shape]
    w = _w(dtype, D, Hq=Hq, Hkv=Hkv, Sq=Sq)
    x = make_inputs(w)
    check(w, run_gpu(w, x).double().cpu().numpy(), run_oracle(w, x), f"{shape} {dtype} D={D}")


@pytest.mark.parametrize("splits", [1, 2, 5, 0])
@pytest.mark.parametrize("shape", ["rows2", "rows16_sq4", "rows17", "rows32_sq2"])
def test_row_counts_splitkv(shape, splits):
    Hq, Hkv, Sq = ROW_SHAPES[shape]
    w = _w(Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=3000, kv_capacity=3000)
    x = make_inputs(w)
    out, lse = run_gpu_splitkv(w, x, splits)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, f"{shape} splits={splits}")
    check_lse(lse.cpu().numpy(), ref_lse, f"{shape} splits={splits} lse", tol=lse_tolerance(w, x))


FEATURES = {
    "dense_noncausal": {"ragged": False, "causal": False, "garbage": None},
    "causal_sq4": {"Sq": 4},
    "window": {"Sq": 2, "local_window": 100},
    "window_noncausal": {"causal": False, "local_window": 64, "ragged": False, "garbage": None},
    "softcap": {"softcap": 2.0, "q_std": 3.0, "k_std": 3.0},
    "mask_per_batch": {"Sq": 3, "mask": "per_batch", "mask_neg_inf_frac": 0.2},
    "mask_per_head": {"Sq": 2, "mask": "per_head", "mask_neg_inf_frac": 0.5},
    "mask_shared_softcap": {"mask": "shared", "mask_neg_inf_frac": 0.1, "softcap": 5.0},
    "all_masked": {"mask": "per_batch", "mask_neg_inf_frac": 1.0},
    "token_major": {"Sq": 3, "out_layout": 1},
    "nonfinite_garbage": {"garbage": "nonfinite", "Sq": 2},
    "short_cache": {"Sk": 70, "kv_capacity": 70},
    "exact_tiles": {"ragged": False, "Sk": 512, "kv_capacity": 512, "garbage": None},
    "scale_override": {"scale": 0.5},
}


@pytest.mark.parametrize("splits", [None, 3])
@pytest.mark.parametrize("feature", list(FEATURES))
def test_features(feature, splits):
    w = _w(**FEATURES[feature])
    x = make_inputs(w)
    if splits is None:
        out = run_gpu(w, x)
        check(w, out.double().cpu().numpy(), run_oracle(w, x), feature)
    else:
        out, lse = run_gpu_splitkv(w, x, splits)
        ref, ref_lse = run_oracle_lse(w, x)
        check(w, out.double().cpu().numpy(), ref, f"{feature} splits={splits}")
        check_lse(lse.cpu().numpy(), ref_lse, f"{feature} splits={splits} lse", tol=lse_tolerance(w, x))


def test_rows_without_keys():
    """Negative past length: the causal limit of the first rows is below 0."""
    w = _w(Sq=4, ragged=False, garbage=None, Sk=300, kv_capacity=300)
    x = make_inputs(w)
    x["total_lengths"] = torch.tensor([300, 2, 150], dtype=torch.int32)
    x["past_lengths"] = torch.tensor([296, -3, 10], dtype=torch.int32)
    out, lse = run_gpu_splitkv(w, x, 2)
    ref, ref_lse = run_oracle_lse(w, x)
    assert np.isneginf(ref_lse[1, :, :2]).all()
    check(w, out.double().cpu().numpy(), ref, "rows without keys")
    check_lse(lse.cpu().numpy(), ref_lse, "rows without keys lse", tol=lse_tolerance(w, x))
    check(w, run_gpu(w, x).double().cpu().numpy(), ref, "rows without keys attn_fwd")


def test_growing_maximum():
    """Keys whose scores grow tile after tile, so the running maximum moves
    by far more than the rescale threshold many times."""
    w = _w(ragged=False, garbage=None, Sk=1024, kv_capacity=1024, causal=False)
    x = make_inputs(w)
    ramp = torch.linspace(0.1, 6.0, w.Sk).view(1, 1, w.Sk, 1)
    x["k"] = (x["k"].float().abs() * ramp).to(x["k"].dtype)
    x["q"] = x["q"].float().abs().to(x["q"].dtype)
    check(w, run_gpu(w, x).double().cpu().numpy(), run_oracle(w, x), "growing maximum")
    out, lse = run_gpu_splitkv(w, x, 4)
    ref, ref_lse = run_oracle_lse(w, x)
    check(w, out.double().cpu().numpy(), ref, "growing maximum split")
    check_lse(lse.cpu().numpy(), ref_lse, "growing maximum lse", tol=lse_tolerance(w, x))


def test_above_32_rows_uses_the_tile_kernel_correctly():
    w = _w(Hq=33, Hkv=1, Sq=1)
    x = make_inputs(w)
    check(w, run_gpu(w, x).double().cpu().numpy(), run_oracle(w, x), "33 rows")


def test_deterministic():
    w = _w(Sq=2, Sk=4000, kv_capacity=4096)
    x = make_inputs(w)
    a, la = run_gpu_splitkv(w, x, 6)
    b, lb = run_gpu_splitkv(w, x, 6)
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert torch.equal(run_gpu(w, x), run_gpu(w, x))


@pytest.mark.parametrize("splits", [0, 1])
def test_full_size_decode_every_row(splits):
    w = EXTRA_WORKLOADS["decode_bf16"]
    x = make_inputs(w)
    ref, ref_lse = run_oracle_lse(w, x)
    if splits == 1:
        out = run_gpu(w, x)
    else:
        out, lse = run_gpu_splitkv(w, x, splits)
        check_lse(lse.cpu().numpy(), ref_lse, "decode_bf16 lse", tol=lse_tolerance(w, x))
    check(w, out.double().cpu().numpy(), ref, f"decode_bf16 splits={splits}, every row")
