"""GPU parity of the fp32 tensor-core entry (attn_fwd_f32_split) against the
fp64 oracle, held to the fp32 path's bound (max abs error <= 1e-4): the DiT
workload scaled down and at full size, the feature matrix and edge cases of
the fp32 CUDA-core path for D = 64 and 128, more work items than CTAs,
garbage cache slots, workspace reuse and the end-to-end host path."""
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from parity import F32_ATOL, check, run_gpu, run_gpu_f32split, run_oracle
from test_parity_gpu import EDGES, FEATURES, MULTI_ITEM, SMALL, _base
from tiled_online_softmax_02_gb300.inputs import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load_library()
    torch.cuda.set_device(0)


def split_check(w, x=None, what=""):
    x = make_inputs(w) if x is None else x
    got = run_gpu_f32split(w, x).double().cpu().numpy()
    return check(w, got, run_oracle(w, x), what or w.name)


@pytest.mark.parametrize("name", ["tiny_f32", "dit_f32"])
def test_workload_small(name):
    split_check(SMALL[name])


@pytest.mark.parametrize("feature", list(FEATURES))
@pytest.mark.parametrize("D", [64, 128])
def test_feature(D, feature):
    split_check(_base("f32", D, **FEATURES[feature]), what=f"f32 split {feature} D={D}")


@pytest.mark.parametrize("edge", list(EDGES))
@pytest.mark.parametrize("D", [64, 128])
def test_edge(D, edge):
    split_check(_base("f32", D, **EDGES[edge]), what=f"f32 split {edge} D={D}")


def test_long_rows_many_tiles():
    """Several 128-row query tiles and dozens of 64-key tiles per row, GQA,
    causal with a ragged tail on both sides."""
    split_check(_base("f32", 128, Hq=8, Hkv=2, Sq=777, Sk=1500, kv_capacity=1600, causal=True))


def test_garbage_slots_do_not_change_output():
    w = _base("f32", 128, ragged=True, Sq=60, Sk=500, kv_capacity=500, causal=True,
              mask="per_batch", mask_neg_inf_frac=0.1, garbage="finite")
    a = make_inputs(w)
    b = dict(a, k=a["k"].clone(), v=a["v"].clone())
    for i, t in enumerate(a["total_lengths"].tolist()):
        b["k"][i, :, t:] = float("nan")
        b["v"][i, :, t:] = float("inf")
    assert torch.equal(run_gpu_f32split(w, a), run_gpu_f32split(w, b))


def test_workspace_reused_across_calls():
    """One workspace, two different problems in a row, then the first again:
    every call rewrites what it reads."""
    w1 = _base("f32", 128, Sq=150, Sk=300, kv_capacity=300, causal=True)
    w2 = _base("f32", 128, ragged=True, Sq=40, Sk=300, kv_capacity=300, causal=True,
               garbage="nonfinite")
    need = attn.load_library().attn_f32_split_workspace_bytes(w1.B, w1.Hkv, 300, 128)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    x1, x2 = make_inputs(w1), make_inputs(w2)
    o1 = run_gpu_f32split(w1, x1, workspace=ws)
    o2 = run_gpu_f32split(w2, x2, workspace=ws)
    o1b = run_gpu_f32split(w1, x1, workspace=ws)
    assert torch.equal(o1, o1b)
    check(w2, o2.double().cpu().numpy(), run_oracle(w2, x2), "second problem")


def test_host_tensors_end_to_end():
    w = SMALL["dit_f32"]
    x = make_inputs(w)
    dev_out = run_gpu_f32split(w, x).cpu()
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    host_out = attn.attn_fwd_f32_split(pin["q"], pin["k"], pin["v"], causal=w.causal,
                                       scale=w.softmax_scale, out_layout=w.out_layout, seq_k=w.Sk)
    assert not host_out.is_cuda
    assert torch.equal(host_out, dev_out)


def test_dit_full_size():
    """The DiT workload at full size (H = 24, S = 1536, D = 128, token-major):
    every element against the oracle, and against the fp32 CUDA-core kernel
    (both within 1e-4 of the exact result)."""
    w = WORKLOADS["dit_f32"]
    x = make_inputs(w)
    out = run_gpu_f32split(w, x)
    check(w, out.double().cpu().numpy(), run_oracle(w, x), "dit_f32 split, full size, every row")
    exact = run_gpu(w, x)
    diff = float((out - exact).abs().max())
    assert diff <= 2 * F32_ATOL, diff


@pytest.mark.parametrize("case", list(MULTI_ITEM))
@pytest.mark.parametrize("D", [64, 128])
def test_more_items_than_ctas(D, case):
    """More 128-row query tiles than CTAs: each persistent CTA runs several
    items, carrying its rings and barrier phases across them."""
    split_check(_base("f32", D, **MULTI_ITEM[case]), what=f"f32 split multi-item {case} D={D}")


def test_split_path_close_to_cuda_core_path():
    """Both fp32 kernels on a masked, soft-capped, windowed ragged problem."""
    w = _base("f32", 64, **FEATURES["everything"])
    x = make_inputs(w)
    a = run_gpu_f32split(w, x)
    b = run_gpu(w, x)
    assert float((a - b).abs().max()) <= 2 * F32_ATOL
