"""GPU parity of the DSA indexer's sparse index selection (dsa_index_select)
against the fp32 oracle: the selected indices must be identical (integer
output) and the fp32 score of every allowed cell, read from the workspace,
bit-identical (the page fixes the score arithmetic and order).  Cases: every
input dtype, head counts on both sides of each register tier, head dims that
are not a multiple of the 32-column chunk, ragged key tails, T = 0, top_k
above / equal to / far above the allowed count, top_k = 1, fully masked rows,
the -1e30 boundary, NaN / inf inputs, exact ties spanning threads, grid-stride
loops, and the full-size prefill and decode workloads: every row's indices
end to end and every allowed score bit-exact on at least 512 rows."""
import numpy as np
import pytest
import torch

import tiled_online_softmax_02_gb300 as attn
from oracle import dsa
from tiled_online_softmax_02_gb300.inputs import DSA_WORKLOADS, DsaWorkload, make_dsa_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load_library()
    torch.cuda.set_device(0)


def _w(**kw) -> DsaWorkload:
    base = dict(name="case", B=2, S=37, H=16, D=64, T=700, top_k=64, dtype="bf16", bias="causal")
    base.update(kw)
    return DsaWorkload(**base)


def run_gpu(w: DsaWorkload, x: dict, ws=None):
    """Indices (numpy int64 [B, 1, S, top_k]) and the workspace tensor."""
    dev = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    if ws is None:
        need = attn.load_library().dsa_index_select_workspace_bytes(w.B, w.S, w.T)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    out = attn.dsa_index_select(dev["query"], dev["key"], dev["weights"], dev["bias"], top_k=w.top_k,
                                scale=w.softmax_scale, weights_scale=w.weights_scale, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ws


def gpu_score_bits(ws, w: DsaWorkload) -> np.ndarray:
    n = w.B * w.S * w.T
    return ws[: n * 4].view(torch.int32).cpu().numpy().view(np.uint32).reshape(w.B, w.S, w.T)


def compare_indices(got: np.ndarray, exp: np.ndarray, what: str):
    assert got.shape == exp.shape, (what, got.shape, exp.shape)
    bad = np.argwhere((got != exp).reshape(-1, got.shape[-1]).any(-1)).reshape(-1)
    if bad.size:
        r = int(bad[0])
        g, e = got.reshape(-1, got.shape[-1])[r], exp.reshape(-1, exp.shape[-1])[r]
        diff = np.flatnonzero(g != e)
        raise AssertionError(f"{what}: {bad.size} rows differ; row {r} first at slot {diff[0]}: "
                             f"gpu {g[diff[:8]]} oracle {e[diff[:8]]}")


def check(w: DsaWorkload, x: dict | None = None, scores: bool = True, what: str = ""):
    x = make_dsa_inputs(w) if x is None else x
    what = what or w.name
    got, ws = run_gpu(w, x)
    args = (x["query"], x["key"], x["weights"], x["bias"])
    kw = dict(scale=w.softmax_scale, weights_scale=w.weights_scale)
    if scores and w.T > 0:
        sc, al = dsa.scores(*args, **kw)
        gb, ob = gpu_score_bits(ws, w), sc.view(np.uint32)
        bad = al.astype(bool) & (gb != ob)
        if bad.any():
            b, s, t = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {int(bad.sum())} score cells differ; first (b={b}, s={s}, t={t}) "
                                 f"gpu {gb[b, s, t]:#010x} oracle {ob[b, s, t]:#010x}")
        exp = dsa.select(sc, al, w.top_k).reshape(w.B, 1, w.S, w.top_k)
    else:
        exp = dsa.index_select(*args, top_k=w.top_k, **kw)
    compare_indices(got, exp, what)
    return got, x


# ---------------------------------------------------------------- dtype x heads x head dim
# D = 64: the TMA-fed tile kernel; D = 60: the general score kernel
@pytest.mark.parametrize("D", [64, 60])
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("H", [1, 7, 16, 17, 32, 33, 64])
def test_heads_and_dtypes(dtype, H, D):
    check(_w(dtype=dtype, H=H, D=D, S=19, T=600, top_k=96, seed=1000 + H), what=f"{dtype} H={H} D={D}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("H", [7, 17, 64])
def test_tile_many_units(dtype, H):
    """Enough (row, key block) units that the tile kernel takes 4 keys a
    lane (small problems take 2); one, two and four head groups."""
    check(_w(dtype=dtype, H=H, D=64, B=1, S=1300, T=600, top_k=50, bias="random", seed=1500 + H),
          what=f"many units {dtype} H={H}")


@pytest.mark.parametrize("D", [1, 16, 31, 32, 33, 48, 100, 128, 192, 256])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_head_dims(D, dtype):
    check(_w(D=D, H=20, S=23, T=530, dtype=dtype, seed=2000 + D), what=f"{dtype} D={D}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_subnormal_products(dtype):
    """Products and partial sums in the fp32 subnormal range: the paired
    instructions must round them like scalar IEEE arithmetic (no flush)."""
    w = _w(dtype=dtype, q_std=3e-20, k_std=2e-19, scale=1.0, weights_scale=1.0, bias="random", seed=2500)
    x = make_dsa_inputs(w)
    x["weights"] = x["weights"] * 1e20            # head terms back in the normal range
    check(w, x, what=f"subnormal {dtype}")


def test_unaligned_query_takes_the_general_path():
    """A query that is not 16-byte aligned must give the same indices (the
    general score kernel) as the aligned one (the tile kernel)."""
    w = _w(D=64, H=8, bias="random", seed=2600)
    x = make_dsa_inputs(w)
    q = x["query"]
    buf = torch.empty(q.numel() + 1, dtype=q.dtype)
    buf[1:].copy_(q.reshape(-1))
    x_off = dict(x, query=buf[1:].view(q.shape))
    assert x_off["query"].data_ptr() % 16 != 0
    got_a, _ = check(w, x, what="aligned")
    got_b, _ = check(w, x_off, what="unaligned")
    assert np.array_equal(got_a, got_b)


@pytest.mark.parametrize("T", [1, 5, 255, 256, 257, 511, 1023])
def test_key_tails(T):
    check(_w(T=T, S=11, top_k=40, bias="random", seed=3000 + T), what=f"T={T}")


@pytest.mark.parametrize("bias", ["causal", "causal_min", "ragged_causal", "random", "zeros"])
def test_bias_modes(bias):
    check(_w(bias=bias, B=3, S=29, T=777, seed=4000), what=bias)


# ---------------------------------------------------------------- top_k edge cases
@pytest.mark.parametrize("top_k", [1, 2, 63, 700, 701, 5000])
def test_top_k(top_k):
    check(_w(top_k=top_k, T=700, bias="random", seed=5000), what=f"top_k={top_k}")


def test_empty_key_axis():
    w = _w(T=0, top_k=9)
    got, _ = check(w, scores=False)
    assert (got == -1).all()


def test_empty_rows():
    w = _w(B=0)
    got, _ = run_gpu(w, make_dsa_inputs(w))
    assert got.shape == (0, 1, w.S, w.top_k)


def test_fully_masked_rows():
    w = _w(bias="random", seed=6000)
    x = make_dsa_inputs(w)
    x["bias"][0, 0, 3] = -np.inf
    x["bias"][1, 0, 7] = -1e30
    x["bias"][1, 0, 8] = float("nan")
    got, _ = check(w, x, what="masked rows")
    assert (got[0, 0, 3] == -1).all() and (got[1, 0, 7] == -1).all() and (got[1, 0, 8] == -1).all()


def test_allow_boundary():
    """bias == -1e30 (as f32) is not allowed; the next f32 above it is; the
    most negative finite f32 and NaN are not; +inf is allowed."""
    w = _w(bias="zeros", top_k=700, seed=6100)
    x = make_dsa_inputs(w)
    m30 = np.float32(-1e30)
    above = np.nextafter(m30, np.float32(0))
    b = x["bias"].numpy()
    b[:, 0, :, 0::5] = m30
    b[:, 0, :, 1::5] = above
    b[:, 0, :, 2::5] = np.finfo(np.float32).min
    b[:, 0, :, 3::5] = np.nan
    b[:, 0, :, 4::10] = np.inf
    got, _ = check(w, x, what="allow boundary")
    sel = got[got >= 0]
    assert set(np.unique(sel % 5)) <= {1, 4}


# ---------------------------------------------------------------- special values and ties
def test_nan_and_inf_inputs():
    w = _w(dtype="f32", bias="random", S=17, T=600, seed=7000)
    x = make_dsa_inputs(w)
    x["weights"][0, 2, 5] = float("nan")          # a NaN weight: the whole row's scores are NaN
    x["weights"][1, 4, 0] = float("inf")          # +inf weight: relu(dot) * inf (NaN where dot <= 0)
    x["weights"][1, 5, 3] = float("-inf")
    x["key"][0, 11] = float("inf")                # an inf key row: inf - inf inside some dots
    x["key"][1, 40, 7] = float("nan")
    x["query"][1, 9, 2, 0] = float("inf")
    x["query"][0, 6, :, :] *= 3e37                # products overflow to inf
    check(w, x, what="nan/inf")


def test_exact_ties_across_threads():
    """All weights zero: every allowed score equals its bias, so with a zero
    bias the whole row ties and the lowest indices win; the tie block spans
    many threads' key ranges."""
    w = _w(bias="zeros", T=3000, top_k=1500, S=5, seed=7100)
    x = make_dsa_inputs(w)
    x["weights"].zero_()
    got, _ = check(w, x, what="all tied")
    assert (got[..., :1500] == np.arange(1500)).all()


def test_duplicate_keys_tie():
    check(_w(ties=True, bias="random", T=1200, top_k=333, seed=7200), what="duplicate keys")


def test_quantised_values_tie():
    """Integer-valued inputs give exactly representable scores with many
    repeats; the radix threshold lands inside large tie groups."""
    w = _w(dtype="f16", bias="zeros", T=2000, top_k=517, S=9, H=5, D=8, seed=7300)
    x = make_dsa_inputs(w)
    g = torch.Generator().manual_seed(7300)
    x["query"] = torch.randint(-2, 3, x["query"].shape, generator=g).to(torch.float16)
    x["key"] = torch.randint(-2, 3, x["key"].shape, generator=g).to(torch.float16)
    x["weights"] = torch.randint(-1, 3, x["weights"].shape, generator=g).to(torch.float16)
    check(w, x, what="quantised ties")


def test_weights_scale_and_scale():
    check(_w(scale=0.37, weights_scale=2.5, seed=7400), what="scales")


# ---------------------------------------------------------------- grid-stride loops, reuse, streams
@pytest.mark.parametrize("D", [8, 64])
def test_many_rows_grid_stride(D):
    """More score units and rows than either kernel's grid holds (D = 8: the
    general score kernel, D = 64: the tile kernel)."""
    check(_w(B=4, S=700, H=2, D=D, T=300, top_k=17, bias="random", seed=8000), what=f"grid stride D={D}")


def test_cluster_ties_across_slices():
    """Few rows: the selection splits each row over a cluster of CTAs; with
    zero weights every allowed key ties, so the lowest-index ties must be
    taken across slice boundaries."""
    w = _w(B=2, S=3, T=3001, top_k=1700, bias="random", seed=8050)
    x = make_dsa_inputs(w)
    x["weights"].zero_()
    x["bias"] = torch.where(torch.isinf(x["bias"]), x["bias"], torch.zeros_like(x["bias"]))
    got, _ = check(w, x, what="cluster ties")
    allowed = (x["bias"].numpy()[:, 0] > np.float32(-1e30))
    for b in range(w.B):
        for s_ in range(w.S):
            exp = np.flatnonzero(allowed[b, s_])[: w.top_k]
            assert np.array_equal(got[b, 0, s_, : exp.size], exp)


def test_long_rows_stream_select():
    """Rows longer than a cluster's shared memory: the streaming selection."""
    check(_w(B=1, S=2, H=1, D=16, T=400_000, top_k=1000, dtype="f32", bias="random", seed=8060),
          what="long rows")


def test_workspace_and_out_reuse_on_side_stream():
    w = _w(bias="random", seed=8100)
    x = make_dsa_inputs(w)
    exp = dsa.index_select(x["query"], x["key"], x["weights"], x["bias"], top_k=w.top_k,
                           scale=w.softmax_scale)
    dev = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    need = attn.load_library().dsa_index_select_workspace_bytes(w.B, w.S, w.T)
    ws = torch.full((need + 64,), 0xAB, dtype=torch.uint8, device="cuda")  # stale counter bytes too
    out = torch.full((w.B, 1, w.S, w.top_k), 12345, dtype=torch.int64, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            attn.dsa_index_select(dev["query"], dev["key"], dev["weights"], dev["bias"], top_k=w.top_k,
                                  scale=w.softmax_scale, out=out, workspace=ws)
    side.synchronize()
    compare_indices(out.cpu().numpy(), exp, "reuse")


def test_host_tensors_end_to_end():
    w = _w(bias="ragged_causal", seed=8200)
    x = make_dsa_inputs(w)
    got = attn.dsa_index_select(x["query"], x["key"], x["weights"], x["bias"], top_k=w.top_k,
                                scale=w.softmax_scale)
    assert got.device.type == "cpu"
    exp = dsa.index_select(x["query"], x["key"], x["weights"], x["bias"], top_k=w.top_k,
                           scale=w.softmax_scale)
    compare_indices(got.numpy(), exp, "host path")


def test_too_many_heads_unsupported():
    w = _w(H=65, T=50, S=2)
    x = make_dsa_inputs(w)
    with pytest.raises(attn.AttnError) as e:
        run_gpu(w, x)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED


# ---------------------------------------------------------------- full size
@pytest.mark.parametrize("name", list(DSA_WORKLOADS))
def test_full_size(name):
    """The full workload in one call: every row's indices against the oracle
    run end to end on that row (threaded over the host cores), and the fp32
    score of every allowed cell bit-exact on at least 512 rows spread over
    the workload (every row when there are fewer)."""
    w = DSA_WORKLOADS[name]
    x = make_dsa_inputs(w)
    got, ws = run_gpu(w, x)
    bits = gpu_score_bits(ws, w)
    kw = dict(scale=w.softmax_scale, weights_scale=w.weights_scale, nthreads=0)
    n_rows = w.B * w.S
    exp = dsa.rows(x["query"], x["key"], x["weights"], x["bias"], np.arange(n_rows), top_k=w.top_k, **kw)
    compare_indices(got.reshape(-1, w.top_k), exp, f"{name} every row end to end")
    rng = np.random.default_rng(9)
    if n_rows <= 512:
        rows = np.arange(n_rows)
    else:
        rows = np.unique(np.concatenate([[0, n_rows - 1], rng.choice(n_rows, size=600, replace=False)]))
    checked = 0
    for b in range(w.B):
        s_idx = rows[rows // w.S == b] % w.S
        if s_idx.size == 0:
            continue
        sc, al = dsa.scores(x["query"][b:b + 1, s_idx], x["key"][b:b + 1], x["weights"][b:b + 1, s_idx],
                            x["bias"][b:b + 1, :, s_idx], **kw)
        ok = al[0].astype(bool)
        gb = bits[b, s_idx]
        bad = ok & (gb != sc.view(np.uint32)[0])
        assert not bad.any(), f"{name}: {int(bad.sum())} score cells differ in batch {b}"
        checked += s_idx.size
    assert checked >= min(512, n_rows)
