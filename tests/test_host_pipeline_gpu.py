"""The end-to-end path with host tensors: the problem is cut into pieces
(one batch, or whole kv-head groups of a batch) whose uploads, kernels and
downloads overlap on three streams.  Each piece is an ordinary call on its
slices, so the host result must equal the device call's bit for bit -- for
every mask broadcast, ragged lengths, GQA groups, both output layouts and the
fp32 tensor-core entry."""
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from tiled_online_softmax_02_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load_library()
    torch.cuda.set_device(0)


CASES = {
    "gqa_causal_two_batches": dict(B=2, Hq=8, Hkv=4, Sq=300, Sk=300, kv_capacity=300, causal=True),
    "one_batch_many_kv_heads": dict(B=1, Hq=16, Hkv=8, Sq=200, Sk=350, kv_capacity=350, causal=True),
    "ragged_mask_per_batch": dict(B=3, Hq=8, Hkv=2, Sq=100, Sk=700, kv_capacity=720, causal=True, ragged=True,
                                  mask="per_batch", mask_neg_inf_frac=0.1, garbage="nonfinite"),
    "mask_per_head_window": dict(B=2, Hq=6, Hkv=3, Sq=150, Sk=400, kv_capacity=400, mask="per_head",
                                 mask_neg_inf_frac=0.2, local_window=100, softcap=10.0),
    "mask_shared": dict(B=4, Hq=4, Hkv=4, Sq=64, Sk=256, kv_capacity=256, mask="shared", causal=True),
    "token_major": dict(B=3, Hq=8, Hkv=2, Sq=120, Sk=120, kv_capacity=120, causal=True, out_layout=1),
    "token_major_one_batch": dict(B=1, Hq=8, Hkv=8, Sq=130, Sk=130, kv_capacity=130, out_layout=1),
    # more batches than pieces: runs of batches, with per-batch mask planes and ragged lengths
    "batch_runs_ragged": dict(B=70, Hq=4, Hkv=2, Sq=40, Sk=96, kv_capacity=100, causal=True, ragged=True,
                              mask="per_batch", mask_neg_inf_frac=0.1),
    "batch_runs_per_head_mask": dict(B=67, Hq=2, Hkv=1, Sq=24, Sk=48, kv_capacity=48, mask="per_head",
                                     out_layout=1),
}


def _call(fn, w, x, **kw):
    return fn(x["q"], x["k"], x["v"], mask=x["mask"], total_lengths=x["total_lengths"],
              past_lengths=x["past_lengths"], causal=w.causal, local_window=w.local_window,
              scale=w.softmax_scale, softcap=w.softcap, out_layout=w.out_layout, seq_k=w.Sk, **kw)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("case", list(CASES))
def test_host_pieces_equal_device_call(case, dtype):
    w = Workload("host", D=128 if dtype != "f16" else 64, dtype=dtype, seed=321, **{"causal": False, **CASES[case]})
    x = make_inputs(w)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    want = _call(attn.attn_fwd, w, dev).cpu()
    got = _call(attn.attn_fwd, w, pin)
    assert not got.is_cuda and torch.equal(got, want)
    if dtype == "f32":  # the fp32 tensor-core entry through the same pieces
        want = _call(attn.attn_fwd_f32_split, w, dev).cpu()
        assert torch.equal(_call(attn.attn_fwd_f32_split, w, pin), want)


def test_unaligned_slices_run_as_one_piece():
    """fp32 with Sq * D not a multiple of four: a head's slice would start
    off the 16-byte alignment, so the host call runs the whole problem as one
    piece -- and still equals the device call."""
    w = Workload("host", B=3, Hq=4, Hkv=2, Sq=37, Sk=51, kv_capacity=53, D=33, dtype="f32", seed=322,
                 causal=True, ragged=True)
    x = make_inputs(w)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    want = _call(attn.attn_fwd, w, dev).cpu()
    assert torch.equal(_call(attn.attn_fwd, w, pin), want)


def test_host_call_rejects_bad_arguments_before_copying():
    w = Workload("host", B=2, Hq=4, Hkv=2, Sq=64, Sk=64, kv_capacity=64, D=128, dtype="bf16", seed=323, causal=False)
    x = make_inputs(w)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = torch.full((2, 4, 64, 128), 7.0, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(attn.AttnError):
        attn.attn_fwd(pin["q"], pin["k"], pin["v"], seq_k=65, out=out)  # Sk > kv_capacity
    with pytest.raises(attn.AttnError):
        attn.attn_fwd(pin["q"], pin["k"], pin["v"], local_window=0, scale=float("nan"), out=out)
    assert bool((out == 7.0).all())  # nothing was written
