"""The allocation-free split-KV entry point (attn_fwd_splitkv_noalloc).

It serves callers that cannot allocate device memory while running attention
(ahead-of-time memory plans, allocation-free execution regions).  Called
through the C ABI, it must give the same result as attn_fwd_splitkv with a
caller-provided workspace, on two calls in a row (the library-owned buffer is
shared and keeps the previous call's contents), and must refuse problems too
large for its buffer.  This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from parity import LP_ATOL, LP_RTOL, check_lse
from tiled_online_softmax_02_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_02_gb300 import build
    build.build()
    torch.cuda.set_device(0)
    return attn.load_library()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, w, g, splits, out, lse):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_fwd_splitkv_noalloc(
        _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]), _ptr(g["mask"]), _ptr(g["total_lengths"]),
        _ptr(g["past_lengths"]), _ptr(out), w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.kv_capacity, w.D,
        int(w.causal), w.local_window, w.softmax_scale, w.softcap, w.out_layout, w.mask_planes,
        attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16, splits, _ptr(lse), stream)


def _reference(w, g, splits):
    return attn.attn_fwd_splitkv(g["q"], g["k"], g["v"], mask=g["mask"],
                                 total_lengths=g["total_lengths"], past_lengths=g["past_lengths"],
                                 causal=w.causal, local_window=w.local_window,
                                 scale=w.softmax_scale, softcap=w.softcap, seq_k=w.Sk,
                                 num_splits=splits)


def _close(got, ref):
    got, ref = got.double().cpu().numpy(), ref.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) <= LP_ATOL + LP_RTOL * np.abs(ref)).all()


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    # decode-like problems: few query rows, long ragged caches, a per-batch mask
    cases = [
        (Workload("noalloc_a", B=2, Hq=8, Hkv=2, Sq=4, Sk=3000, kv_capacity=3072, D=128,
                  dtype="bf16", causal=True, ragged=True, garbage="nonfinite", mask="per_batch",
                  mask_neg_inf_frac=0.1, seed=91), 8),
        (Workload("noalloc_b", B=3, Hq=4, Hkv=4, Sq=1, Sk=2500, kv_capacity=2500, D=64,
                  dtype="f16", causal=True, seed=92), 0),
    ]
    for w, splits in cases:
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(w).items()}
        ref_out, ref_lse = _reference(w, g, splits)
        torch.cuda.synchronize()
        out = torch.empty_like(ref_out)
        lse = torch.empty_like(ref_lse)
        assert _noalloc(lib, w, g, splits, out, lse) == attn.ATTN_OK
        torch.cuda.synchronize()
        assert attn.get_device_status() == attn.ATTN_OK
        _close(out, ref_out)
        check_lse(lse.cpu().numpy(), ref_lse.cpu().numpy(), f"{w.name} lse")


def test_noalloc_refuses_problems_beyond_its_buffer(lib):
    w = Workload("noalloc_big", B=8, Hq=32, Hkv=4, Sq=128, Sk=4096, kv_capacity=4096, D=128,
                 dtype="f16", causal=True, seed=93)
    need = lib.attn_splitkv_workspace_bytes(w.B, w.Hq, w.Sq, w.D, 4)
    assert need > 8 << 20
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in make_inputs(w).items()}
    out = torch.full((w.B, w.Hq, w.Sq, w.D), 3.0, dtype=torch.float16, device="cuda")
    assert _noalloc(lib, w, g, 4, out, None) == attn.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())  # nothing was launched
