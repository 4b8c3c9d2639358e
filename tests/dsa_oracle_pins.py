"""Pins of the DSA indexer oracle (oracle/dsa_oracle.c) to facts outside it.

Source: "onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/dsa_index_select.rs",
module doc and score kernel: score = sum over heads (ascending) of
relu(scale * q_h . k) * (w_h * weights_scale), dot products over head_dim
ascending, every multiply and add rounded to fp32 separately, plus the f32
bias; allowed iff bias > -1e30; the top min(#allowed, top_k) by (score desc,
index asc) in f32 total order with NaN canonicalised to +NaN; emitted
ascending, padded with -1.

Each pin takes a loaded oracle library and raises AssertionError on a
mismatch.  What pins it:
  - exact arithmetic: small integer inputs make every fp32 step exact, so
    the scores equal numpy's float64 einsum of the same formula;
  - the page's operation order, where fp32 rounding depends on it: the dot
    product left to right over head_dim, the head sum left to right, and no
    fused multiply-add (values worked by hand below);
  - the allow rule at and around -1e30, and +/-inf biases;
  - selection against numpy's stable sort, ties to the lowest index, the -1
    padding, ascending output, -0 below +0, NaN above +inf;
  - ReLU, weights_scale, batch indexing of the key, permutation of keys.
"""
from __future__ import annotations

import numpy as np

from oracle import dsa

F32 = np.float32


def _idx(lib, q, k, w, bias, top_k, scale, ws=1.0):
    return dsa.index_select(q, k, w, bias, top_k=top_k, scale=scale, weights_scale=ws, lib=lib)


def _expected_exact(q, k, w, bias, scale, ws):
    """float64 reference of the score for inputs where fp32 is exact."""
    dots = np.einsum("bshd,btd->bsht", q.astype(np.float64), k.astype(np.float64))
    scored = np.maximum(scale * dots, 0.0)
    weighted = np.einsum("bsht,bsh->bst", scored, w.astype(np.float64) * ws)
    return weighted + bias[:, 0].astype(np.float64)


def pin_exact_integer_scores(lib):
    rng = np.random.default_rng(11)
    B, S, H, D, T = 2, 3, 3, 8, 10
    q = rng.integers(-3, 4, (B, S, H, D)).astype(F32)
    k = rng.integers(-3, 4, (B, T, D)).astype(F32)
    w = rng.integers(-2, 3, (B, S, H)).astype(F32)
    bias = rng.integers(-4, 5, (B, 1, S, T)).astype(F32)
    bias[0, 0, 1, 4] = -np.inf
    scale, ws = 0.5, 2.0
    sc, al = dsa.scores(q, k, w, bias, scale=scale, weights_scale=ws, lib=lib)
    exp = _expected_exact(q, k, w, bias, scale, ws)
    assert al[0, 1, 4] == 0 and sc[0, 1, 4] == -np.inf
    m = al.astype(bool)
    assert np.array_equal(sc[m].astype(np.float64), exp[m]), "exact integer scores"


def pin_dot_order_left_to_right(lib):
    # terms 2^24, 1, -2^24 over d ascending: (2^24 + 1) rounds to 2^24 (tie to
    # even), then -2^24 gives 0; any other order gives 1
    q = np.array([[[[2.0 ** 24, 1.0, -(2.0 ** 24)]]]], dtype=F32)
    k = np.ones((1, 1, 3), dtype=F32)
    w = np.ones((1, 1, 1), dtype=F32)
    bias = np.zeros((1, 1, 1, 1), dtype=F32)
    sc, _ = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    assert sc[0, 0, 0] == 0.0, f"dot order: {sc[0, 0, 0]}"


def pin_head_sum_left_to_right(lib):
    # per-head terms 2^24, 1, 1: ((2^24 + 1) + 1) stays 2^24; 1 + 1 first would give 2^24 + 2
    q = np.array([[[[2.0 ** 24], [1.0], [1.0]]]], dtype=F32)  # [1,1,3,1]
    k = np.ones((1, 1, 1), dtype=F32)
    w = np.ones((1, 1, 3), dtype=F32)
    bias = np.zeros((1, 1, 1, 1), dtype=F32)
    sc, _ = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    assert sc[0, 0, 0] == F32(2.0 ** 24), f"head order: {sc[0, 0, 0]}"


def pin_no_fused_multiply_add(lib):
    # a = 1 + 2^-12: a * a = 1 + 2^-11 + 2^-24 rounds to 1 + 2^-11 (tie to
    # even).  Added to a running sum of -(1 + 2^-11), the rounded product gives
    # exactly 0; a fused multiply-add keeps the 2^-24.
    a = F32(1.0 + 2.0 ** -12)
    c = F32(1.0 + 2.0 ** -11)
    # in the dot product: terms -(1 + 2^-11) (exact) then a * a
    q = np.array([[[[-c, a]]]], dtype=F32)
    k = np.array([[[1.0, a]]], dtype=F32)
    w = np.ones((1, 1, 1), dtype=F32)
    bias = np.zeros((1, 1, 1, 1), dtype=F32)
    sc, _ = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    assert sc[0, 0, 0] == 0.0, f"fused multiply-add in the dot product: {sc[0, 0, 0]!r}"
    # in the head sum: head 0 adds c * -1 = -(1 + 2^-11), head 1 adds a * a
    q2 = np.array([[[[c], [a]]]], dtype=F32)   # dots c and a (one key of 1)
    k2 = np.ones((1, 1, 1), dtype=F32)
    w2 = np.array([[[-1.0, a]]], dtype=F32)
    sc2, _ = dsa.scores(q2, k2, w2, bias, scale=1.0, lib=lib)
    assert sc2[0, 0, 0] == 0.0, f"fused multiply-add in the head sum: {sc2[0, 0, 0]!r}"


def pin_allow_threshold(lib):
    T = 6
    q = np.ones((1, 1, 1, 2), dtype=F32)
    k = np.ones((1, T, 2), dtype=F32)
    w = np.ones((1, 1, 1), dtype=F32)
    bias = np.array([[[[-1e30, -9.9e29, -np.inf, np.inf, 0.0, -3.4e38]]]], dtype=F32)
    sc, al = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    assert list(al[0, 0]) == [0, 1, 0, 1, 1, 0], list(al[0, 0])
    assert sc[0, 0, 3] == np.inf
    out = _idx(lib, q, k, w, bias, 5, 1.0)
    assert list(out[0, 0, 0]) == [1, 3, 4, -1, -1], list(out[0, 0, 0])


def pin_selection_matches_numpy_sort(lib):
    rng = np.random.default_rng(12)
    rows, T = 7, 300
    sc = rng.standard_normal((rows, T)).astype(F32)
    al = (rng.random((rows, T)) > 0.3).astype(np.uint8)
    al[3] = 0
    al[4, :5] = 1
    al[4, 5:] = 0
    for top_k in (1, 17, 128, 400):
        out = dsa.select(sc, al, top_k, lib=lib)
        for r in range(rows):
            cand = np.nonzero(al[r])[0]
            order = cand[np.argsort(-sc[r, cand].astype(np.float64), kind="stable")]
            keep = min(len(cand), top_k)
            exp = np.full(top_k, -1, dtype=np.int64)
            exp[:keep] = np.sort(order[:keep])
            assert np.array_equal(out[r], exp), (r, top_k)


def pin_ties_go_to_lowest_index(lib):
    sc = np.array([[1.0, 5.0, 3.0, 5.0, 5.0, 2.0, 5.0]], dtype=F32)
    al = np.ones_like(sc, dtype=np.uint8)
    assert list(dsa.select(sc, al, 3, lib=lib)[0]) == [1, 3, 4]
    assert list(dsa.select(sc, al, 2, lib=lib)[0]) == [1, 3]


def pin_total_order_specials(lib):
    nan = np.float32(np.nan)
    sc = np.array([[-0.0, 0.0, -np.inf, np.inf, nan, 7.0]], dtype=F32)
    al = np.ones_like(sc, dtype=np.uint8)
    assert list(dsa.select(sc, al, 1, lib=lib)[0]) == [4]           # +NaN above +inf
    assert list(dsa.select(sc, al, 2, lib=lib)[0]) == [3, 4]
    assert list(dsa.select(sc, al, 3, lib=lib)[0]) == [3, 4, 5]
    assert list(dsa.select(sc, al, 4, lib=lib)[0]) == [1, 3, 4, 5]  # +0 before -0
    assert list(dsa.select(sc, al, 6, lib=lib)[0]) == [0, 1, 2, 3, 4, 5]


def pin_nan_score_is_canonical_and_first(lib):
    # w = inf makes 0 * inf = NaN on a head whose dot is negative -> the cell's
    # score is NaN, canonicalised to +NaN, and ranks above everything
    q = np.array([[[[1.0, 0.0], [-1.0, 0.0]]]], dtype=F32)  # heads: +k0, -k0
    k = np.array([[[1.0, 0.0], [2.0, 0.0], [3.0, 0.0]]], dtype=F32)
    w = np.array([[[1.0, np.inf]]], dtype=F32)
    bias = np.zeros((1, 1, 1, 3), dtype=F32)
    sc, _ = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    assert np.isnan(sc).all()
    bits = sc.view(np.uint32)
    assert (bits == 0x7FC00000).all(), [hex(b) for b in bits.ravel()]
    # with finite weights instead, the top key is the largest dot
    w2 = np.array([[[1.0, 5.0]]], dtype=F32)
    assert list(_idx(lib, q, k, w2, bias, 1, 1.0)[0, 0, 0]) == [2]


def pin_relu_and_weights_scale(lib):
    # head 1 has a negative dot with every key: ReLU drops it whatever its weight
    q = np.array([[[[1.0, 0.0], [0.0, -1.0]]]], dtype=F32)
    k = np.array([[[1.0, 2.0], [3.0, 1.0]]], dtype=F32)
    w = np.array([[[2.0, 100.0]]], dtype=F32)
    bias = np.array([[[[0.5, -0.5]]]], dtype=F32)
    sc, _ = dsa.scores(q, k, w, bias, scale=0.25, weights_scale=4.0, lib=lib)
    assert sc[0, 0, 0] == F32(0.25 * 1.0 * 8.0 + 0.5), sc
    assert sc[0, 0, 1] == F32(0.25 * 3.0 * 8.0 - 0.5), sc


def pin_key_batch_indexing_and_permutation(lib):
    rng = np.random.default_rng(13)
    B, S, H, D, T = 3, 2, 2, 4, 9
    q = rng.integers(-2, 3, (B, S, H, D)).astype(F32)
    k = rng.integers(-2, 3, (B, T, D)).astype(F32)
    w = rng.integers(1, 3, (B, S, H)).astype(F32)
    bias = (np.arange(T, dtype=F32) * F32(1e-3))[None, None, None, :].repeat(B, 0).repeat(S, 2)
    sc, _ = dsa.scores(q, k, w, bias, scale=1.0, lib=lib)
    exp = _expected_exact(q, k, w, np.zeros_like(bias), 1.0, 1.0)
    assert np.allclose(sc.astype(np.float64) - bias[:, 0].astype(np.float64), exp, atol=1e-6)
    # permuting the keys (and their bias) permutes the selected positions
    perm = rng.permutation(T)
    out = _idx(lib, q, k, w, bias, 4, 1.0)
    out_p = _idx(lib, q, k[:, perm], w, bias[..., perm], 4, 1.0)
    inv = np.argsort(perm)
    for b in range(B):
        for s in range(S):
            a = sorted(int(i) for i in out[b, 0, s] if i >= 0)
            c = sorted(int(perm[i]) for i in out_p[b, 0, s] if i >= 0)
            assert a == c, (b, s)
    assert inv is not None


def pin_rows_equal_full(lib):
    rng = np.random.default_rng(14)
    B, S, H, D, T = 2, 5, 4, 16, 40
    q = rng.standard_normal((B, S, H, D)).astype(F32)
    k = rng.standard_normal((B, T, D)).astype(F32)
    w = rng.standard_normal((B, S, H)).astype(F32)
    bias = np.where(rng.random((B, 1, S, T)) < 0.2, -np.inf, 0.0).astype(F32)
    bias[0, 0, 3, 5:9] = F32(-1e30)    # exactly at the threshold: not allowed
    bias[1, 0, 4, 2] = F32(-9.9e29)    # just above it: allowed
    rows = np.array([0, 3, 7, 9])
    for top_k in (12, T):  # top_k = T lists every allowed key
        full = _idx(lib, q, k, w, bias, top_k, 0.125)
        part = dsa.rows(q, k, w, bias, rows, top_k=top_k, scale=0.125, lib=lib)
        assert np.array_equal(part, full.reshape(B * S, top_k)[rows])
    assert full[0, 0, 3, :].tolist().count(5) == 0  # at the threshold: never listed


def pin_threaded_calls_equal_one_thread(lib):
    """Splitting rows over threads changes nothing: bit-identical scores and
    identical indices, for row chunks that cross batch boundaries."""
    rng = np.random.default_rng(15)
    B, S, H, D, T = 3, 7, 5, 24, 50
    q = rng.standard_normal((B, S, H, D)).astype(F32)
    k = rng.standard_normal((B, T, D)).astype(F32)
    w = rng.standard_normal((B, S, H)).astype(F32)
    bias = np.where(rng.random((B, 1, S, T)) < 0.3, -np.inf, rng.standard_normal((B, 1, S, T))).astype(F32)
    sc1, al1 = dsa.scores(q, k, w, bias, scale=0.2, lib=lib)
    for nt in (2, 4, 0):
        scn, aln = dsa.scores(q, k, w, bias, scale=0.2, nthreads=nt, lib=lib)
        assert np.array_equal(sc1.view(np.uint32), scn.view(np.uint32)) and np.array_equal(al1, aln)
        rows = np.arange(B * S)[::-1].copy()
        r1 = dsa.rows(q, k, w, bias, rows, top_k=9, scale=0.2, lib=lib)
        rn = dsa.rows(q, k, w, bias, rows, top_k=9, scale=0.2, nthreads=nt, lib=lib)
        assert np.array_equal(r1, rn)


PINS = [v for name, v in sorted(globals().items()) if name.startswith("pin_") and callable(v)]
