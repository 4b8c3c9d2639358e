"""Entry points captured into CUDA graphs.  A call allocates and synchronises
nothing, so it can be captured; the split-KV merge and the DSA selection are
programmatic dependents of the kernel before them, which capture turns into
programmatic graph edges.  Replaying the graph must give the same bits as a
direct call on the same inputs, and again on a second replay (the DSA unit
counter is re-zeroed by the captured memset)."""
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from parity import to_dev
from tiled_online_softmax_02_gb300.inputs import (DSA_WORKLOADS, EXTRA_WORKLOADS, WORKLOADS, Workload,
                                                  make_dsa_inputs, make_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tiled_online_softmax_02_gb300 import build
    build.build()
    attn.load_library()
    torch.cuda.set_device(0)


def _capture(fn):
    """fn once on a side stream (first-call setup happens outside the
    capture), then captured into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _replay_twice(g, outs, refs):
    for _ in range(2):
        for o in outs:
            o.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert attn.get_device_status() == attn.ATTN_OK
        for o, r in zip(outs, refs):
            assert torch.equal(o, r)


@pytest.mark.parametrize("name,shape", [
    ("decode_clusters", dict(T=8192)),                     # 8 rows: selection over clusters of CTAs
    ("prefill_rows", dict(S=384, T=384, top_k=96)),        # one CTA a row
])
def test_dsa_index_select_graph(name, shape):
    base = "dsa_decode_bf16" if name.startswith("decode") else "dsa_prefill_bf16"
    w = DSA_WORKLOADS[base].replace(**shape)
    x = make_dsa_inputs(w)
    q, k, wt, b = (x[n].cuda() for n in ("query", "key", "weights", "bias"))
    kw = dict(top_k=w.top_k, scale=w.softmax_scale, weights_scale=w.weights_scale)
    ref = attn.dsa_index_select(q, k, wt, b, **kw)
    lib = attn.load_library()
    ws = torch.empty(lib.dsa_index_select_workspace_bytes(w.B, w.S, w.T), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    g = _capture(lambda: attn.dsa_index_select(q, k, wt, b, out=out, workspace=ws, **kw))
    _replay_twice(g, [out], [ref])


@pytest.mark.parametrize("name,kw", [
    ("decode", dict()),
    ("chunk_prefill_mask", dict(Sq=100, ragged=True, Sk=1200, kv_capacity=1200, mask="per_batch",
                                mask_neg_inf_frac=0.1, garbage="finite")),
])
def test_splitkv_graph(name, kw):
    w = Workload("splitkv_graph", B=2, Hq=8, Hkv=2, Sq=1, Sk=1500, kv_capacity=1500, D=128, dtype="bf16",
                 causal=True, seed=4322).replace(**kw)
    g_in = to_dev(make_inputs(w))
    args = dict(mask=g_in["mask"], total_lengths=g_in["total_lengths"], past_lengths=g_in["past_lengths"],
                causal=w.causal, local_window=w.local_window, scale=w.softmax_scale, softcap=w.softcap,
                out_layout=w.out_layout, seq_k=w.Sk, num_splits=4)
    ref_o, ref_l = attn.attn_fwd_splitkv(g_in["q"], g_in["k"], g_in["v"], **args)
    lib = attn.load_library()
    ws = torch.empty(lib.attn_splitkv_workspace_bytes(w.B, w.Hq, w.Sq, w.D, 4) // 4, dtype=torch.float32,
                     device="cuda")
    out, lse = torch.empty_like(ref_o), torch.empty_like(ref_l)
    g = _capture(lambda: attn.attn_fwd_splitkv(g_in["q"], g_in["k"], g_in["v"], out=out, lse=lse,
                                               workspace=ws, **args))
    _replay_twice(g, [out, lse], [ref_o, ref_l])


@pytest.mark.parametrize("name,kw", [
    ("gqa_causal_bf16", dict(B=1, Hq=4, Hkv=2, Sq=300, Sk=300, kv_capacity=300)),
    ("decode_bf16", dict(B=2, Sk=3000, kv_capacity=3072)),  # the decode kernel, clusters merging on chip
])
def test_attn_fwd_graph(name, kw):
    w = {**WORKLOADS, **EXTRA_WORKLOADS}[name].replace(**kw)
    g_in = to_dev(make_inputs(w))
    args = dict(mask=g_in["mask"], total_lengths=g_in["total_lengths"], past_lengths=g_in["past_lengths"],
                causal=w.causal, local_window=w.local_window, scale=w.softmax_scale, softcap=w.softcap,
                out_layout=w.out_layout, seq_k=w.Sk)
    ref = attn.attn_fwd(g_in["q"], g_in["k"], g_in["v"], **args)
    out = torch.empty_like(ref)
    g = _capture(lambda: attn.attn_fwd(g_in["q"], g_in["k"], g_in["v"], out=out, **args))
    _replay_twice(g, [out], [ref])


@pytest.mark.parametrize("kw", [
    dict(B=1, Hq=4, Hkv=4, Sq=300, Sk=300, kv_capacity=300, D=128),
    dict(B=2, Hq=4, Hkv=2, Sq=200, Sk=260, kv_capacity=272, D=64, causal=True, ragged=True, garbage="nonfinite"),
])
def test_f32_split_graph(kw):
    """fp32 on the tensor cores: the attention kernel is a programmatic
    dependent of the K / V pre-pass (it starts its prologue and Q rows during
    the pre-pass and waits for it before reading the pieces)."""
    w = WORKLOADS["dit_f32"].replace(**kw)
    g_in = to_dev(make_inputs(w))
    args = dict(mask=g_in["mask"], total_lengths=g_in["total_lengths"], past_lengths=g_in["past_lengths"],
                causal=w.causal, local_window=w.local_window, scale=w.softmax_scale, softcap=w.softcap,
                out_layout=w.out_layout, seq_k=w.Sk)
    ref = attn.attn_fwd_f32_split(g_in["q"], g_in["k"], g_in["v"], **args)
    lib = attn.load_library()
    ws = torch.empty(max(lib.attn_f32_split_workspace_bytes(w.B, w.Hkv, w.kv_capacity, w.D), 16),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(ref)
    g = _capture(lambda: attn.attn_fwd_f32_split(g_in["q"], g_in["k"], g_in["v"], out=out, workspace=ws, **args))
    _replay_twice(g, [out], [ref])
