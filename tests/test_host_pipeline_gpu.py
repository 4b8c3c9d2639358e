"""The end-to-end path with host tensors: the problem is cut into pieces
(one batch, or whole kv-head groups of a batch) whose uploads, kernels and
downloads overlap on three streams.  Each piece is an ordinary call on its
slices, so the host result must equal the device call's bit for bit -- for
every mask broadcast, ragged lengths, GQA groups, both output layouts and the
fp32 tensor-core entry."""
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from tiled_online_softmax_02_gb300 import _binding
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


NAN_CASES = {
    "ragged_per_batch_mask": dict(B=3, Hq=8, Hkv=2, Sq=100, Sk=700, kv_capacity=720, causal=True, ragged=True,
                                  mask="per_batch", mask_neg_inf_frac=0.1),
    "ragged_per_head_mask": dict(B=2, Hq=4, Hkv=4, Sq=64, Sk=300, kv_capacity=300, causal=True, ragged=True,
                                 mask="per_head", mask_neg_inf_frac=0.1),
    "ragged_shared_mask_window": dict(B=4, Hq=4, Hkv=2, Sq=40, Sk=500, kv_capacity=512, ragged=True,
                                      mask="shared", local_window=64, out_layout=1),
    "seq_k_below_capacity": dict(B=2, Hq=4, Hkv=1, Sq=90, Sk=200, kv_capacity=256, causal=True),
}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("case", list(NAN_CASES))
def test_slots_past_the_valid_keys_are_not_uploaded(case, dtype):
    """attn_fwd_host uploads only cache rows and mask columns j < min(lsk, Sk):
    with every device buffer first filled with NaN, the output still equals
    the device call on fully uploaded inputs, and the bytes it reports are
    exactly those rows and columns plus q and the lengths."""
    import ctypes
    w = Workload("host", D=128 if dtype == "bf16" else 64, dtype=dtype, seed=324,
                 **{"causal": False, **NAN_CASES[case]})
    x = make_inputs(w)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    want = _call(attn.attn_fwd, w, dev).cpu()
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    d = {}
    for name in ("q", "k", "v", "mask"):
        t = x[name]
        d[name] = None if t is None else torch.full(t.shape, float("nan"), dtype=t.dtype, device="cuda")
    for name in ("total_lengths", "past_lengths"):
        t = x[name]
        d[name] = None if t is None else torch.full(t.shape, -7, dtype=torch.int32, device="cuda")
    dout = torch.full(want.shape, float("nan"), dtype=want.dtype, device="cuda")
    host_out = torch.empty(want.shape, dtype=want.dtype).pin_memory()
    lib = attn.load_library()
    copied = (ctypes.c_uint64 * 2)()
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    torch.cuda.synchronize()
    rc = lib.attn_fwd_host(ptr(pin["q"]), ptr(pin["k"]), ptr(pin["v"]), ptr(pin["mask"]),
                           ptr(pin["total_lengths"]), ptr(pin["past_lengths"]), ptr(host_out),
                           ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["mask"]), ptr(d["total_lengths"]),
                           ptr(d["past_lengths"]), ptr(dout), w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.kv_capacity, w.D,
                           int(w.causal), w.local_window, w.softmax_scale, w.softcap, w.out_layout,
                           0 if x["mask"] is None else x["mask"].shape[0], _binding.DTYPE_CODES[x["q"].dtype],
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), copied)
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    assert torch.equal(host_out, want)
    # the bytes the header's rule gives
    es = x["q"].element_size()
    tot = x["total_lengths"]
    rows = [min(max(int(tot[b]), 0), w.Sk) if tot is not None else w.Sk for b in range(w.B)]
    up = x["q"].numel() * es + 2 * sum(rows) * w.Hkv * w.D * es
    up += sum(4 * t.numel() for t in (x["total_lengths"], x["past_lengths"]) if t is not None)
    if w.mask == "per_batch":
        up += sum(rows) * w.Sq * 4
    elif w.mask == "per_head":
        up += sum(rows) * w.Hq * w.Sq * 4
    elif w.mask == "shared":
        up += max(rows) * w.Sq * 4
    assert (copied[0], copied[1]) == (up, want.numel() * es)
    assert sum(rows) < w.B * w.kv_capacity  # the case leaves slots out
