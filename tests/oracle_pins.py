"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle library handle (``oracle.load()`` or a
deliberately broken variant built by the mutation test) and raises
AssertionError when the oracle disagrees with:

* hand-worked closed forms (``tests/golden/closed_form_cases.txt``),
* PyTorch's own CPU scaled-dot-product attention in float64 (a library
  routine) on the cases it covers (causal, boolean / additive masks, GQA),
* the pages' two streaming recurrences, re-derived here in fp64: the
  16-key tile update of "onnx-runtime-ep-cuda 0.1.0-dev.5,
  src/kernels/flash_attention.rs" (`flash_attention_body`: tile max, tile sum,
  alpha / beta rescale) and the per-key update of "pictor-kernels 0.1.0,
  src/gpu_backend/cuda_imagen_attn_kernels.rs" (module doc "Kernel
  structure"),
* invariants and special cases of the definition (uniform V, shift
  invariance of a mask row, -inf mask = deleted key, window 1, huge window,
  huge soft-cap, GQA = replicated MHA, ragged = sliced dense, garbage slots,
  token-major = transposed head-major).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "closed_form_cases.txt")


# ----------------------------------------------------------------- helpers
def _run(lib, q, k, v, *, causal=False, local_window=0, scale=None, softcap=0.0,
         out_layout=0, mask=None, mask_planes=0, total=None, past=None, Sk=None):
    q = np.asarray(q, dtype=np.float32)
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    B, Hq, Sq, D = q.shape
    Hkv, cap = k.shape[1], k.shape[2]
    Sk = cap if Sk is None else Sk
    return oracle.attn_fwd(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, kv_capacity=cap, D=D,
                           causal=causal, local_window=local_window, scale=scale,
                           softcap=softcap, out_layout=out_layout, mask=mask,
                           mask_planes=mask_planes, total_lengths=total, past_lengths=past,
                           nthreads=2, lib=lib)


def _rand(rng, *shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


def parse_golden(path: str = GOLDEN) -> list[dict]:
    env = {"e": math.e, "exp": math.exp, "tanh": math.tanh, "log": math.log,
           "inf": math.inf, "__builtins__": {}}
    cases, cur = [], {}
    for raw in open(path).read().splitlines() + [""]:
        line = raw.strip()
        if line.startswith("#"):
            continue
        if not line:
            if cur:
                cases.append(cur)
                cur = {}
            continue
        key, _, val = line.partition(":")
        key, val = key.strip(), val.strip()
        if key in ("shape", "flags"):
            for tok in val.split():
                name, _, num = tok.partition("=")
                cur[name] = float(num) if "." in num else int(num)
        elif key == "name":
            cur["name"] = val
        else:
            cur[key] = eval(val, env)  # noqa: S307 - fixture expressions: numbers and e/exp/tanh/log
    return cases


# ------------------------------------------------------------------- pins
def pin_closed_forms(lib):
    for c in parse_golden():
        got = _run(lib, c["q"], c["k"], c["v"], causal=bool(c["causal"]),
                   local_window=c["local_window"], scale=float(c["scale"]),
                   softcap=float(c["softcap"]), out_layout=c["out_layout"],
                   mask=c.get("mask"), mask_planes=c["mask_planes"],
                   total=c.get("total_lengths"), past=c.get("past_lengths"), Sk=c["Sk"])
        _close(got, c["expected"], 1e-13, c["name"])


def _torch_sdpa(q, k, v, *, bool_mask=None, add_mask=None, scale):
    """PyTorch CPU float64 SDPA; K/V heads expanded for GQA."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))
    kt = torch.from_numpy(np.asarray(k, dtype=np.float64))
    vt = torch.from_numpy(np.asarray(v, dtype=np.float64))
    g = qt.shape[1] // kt.shape[1]
    kt = kt.repeat_interleave(g, dim=1)
    vt = vt.repeat_interleave(g, dim=1)
    m = None
    if bool_mask is not None:
        m = torch.from_numpy(bool_mask)
    if add_mask is not None:
        am = torch.from_numpy(np.asarray(add_mask, dtype=np.float64))
        m = am if m is None else am.masked_fill(~m, -math.inf)
    return F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale).numpy()


def pin_torch_sdpa(lib):
    rng = np.random.default_rng(11)
    for (B, Hq, Hkv, Sq, Sk, D) in [(2, 4, 2, 5, 9, 8), (1, 3, 1, 7, 7, 16), (2, 2, 2, 1, 6, 4),
                                    (1, 8, 2, 33, 70, 32)]:
        q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
        scale = 0.3 + rng.random()
        # non-causal, no mask
        _close(_run(lib, q, k, v, scale=scale), _torch_sdpa(q, k, v, scale=scale), 1e-12,
               f"sdpa plain {B,Hq,Hkv,Sq,Sk,D}")
        # causal, bottom-right aligned (key j visible iff j <= Sk - Sq + qi)
        tri = np.tril(np.ones((Sq, Sk), dtype=bool), k=Sk - Sq)
        _close(_run(lib, q, k, v, causal=True, scale=scale),
               _torch_sdpa(q, k, v, bool_mask=tri, scale=scale), 1e-12,
               f"sdpa causal {B,Hq,Hkv,Sq,Sk,D}")
        # additive per-(batch, head) mask, no -inf so no row is empty
        am = _rand(rng, B, Hq, Sq, Sk)
        _close(_run(lib, q, k, v, scale=scale, mask=am.reshape(B * Hq, Sq, Sk),
                    mask_planes=B * Hq),
               _torch_sdpa(q, k, v, add_mask=am, scale=scale), 1e-12,
               f"sdpa additive {B,Hq,Hkv,Sq,Sk,D}")
        # additive mask + causal together
        _close(_run(lib, q, k, v, causal=True, scale=scale, mask=am.reshape(B * Hq, Sq, Sk),
                    mask_planes=B * Hq),
               _torch_sdpa(q, k, v, bool_mask=tri, add_mask=am, scale=scale), 1e-12,
               f"sdpa causal+additive {B,Hq,Hkv,Sq,Sk,D}")


def _stream_tiles(q, k, v, vis_bias, scale, tile):
    """fp64 re-derivation of the tile-wise online-softmax update: per tile the
    tile max m_t and tile sum t of exp(s - m_t); an all-masked tile changes
    nothing; otherwise m' = max(m, m_t) (m_t on the first live tile),
    alpha = exp(m - m'), beta = exp(m_t - m'), l' = alpha l + beta t,
    O' = alpha O + beta sum exp(s - m_t) v.  vis_bias[j] is 0 or -inf (plus
    the additive mask)."""
    Sk, D = k.shape
    m, l, o = -math.inf, 0.0, np.zeros(D)
    for k0 in range(0, Sk, tile):
        s = scale * (k[k0:k0 + tile] @ q) + vis_bias[k0:k0 + tile]
        mt = s.max()
        if mt == -math.inf:
            continue
        e = np.where(np.isneginf(s), 0.0, np.exp(s - mt))
        t = e.sum()
        mn = max(m, mt) if l > 0 else mt
        alpha = math.exp(m - mn) if l > 0 else 0.0
        beta = math.exp(mt - mn)
        l = alpha * l + beta * t
        o = alpha * o + beta * (e @ v[k0:k0 + tile])
        m = mn
    return o / l if l > 0 else np.zeros(D)


def _stream_keys(q, k, v, vis_bias, scale):
    """fp64 re-derivation of the per-key online update: m' = max(m, s),
    c = exp(m - m') (0 on the first key), p = exp(s - m'), l = l c + p,
    O = O c + p v."""
    m, l, o = -math.inf, 0.0, np.zeros(k.shape[1])
    for j in range(k.shape[0]):
        s = scale * float(k[j] @ q) + vis_bias[j]
        if s == -math.inf:
            continue
        mn = max(m, s)
        c = 0.0 if m == -math.inf else math.exp(m - mn)
        p = math.exp(s - mn)
        l = l * c + p
        o = o * c + p * v[j]
        m = mn
    return o / l if l > 0 else np.zeros(k.shape[1])


def pin_streaming_recurrences(lib):
    rng = np.random.default_rng(12)
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 1, 9, 53, 8
    q, k, v = _rand(rng, B, Hq, Sq, D, std=2.0), _rand(rng, B, Hkv, Sk, D, std=2.0), \
        _rand(rng, B, Hkv, Sk, D)
    am = _rand(rng, 1, Sq, Sk)
    am[rng.random(am.shape) < 0.2] = -np.inf
    am[0, 3, :] = -np.inf  # one fully masked row
    scale = 0.4
    got = _run(lib, q, k, v, causal=True, scale=scale, mask=am, mask_planes=1)
    for h in range(Hq):
        for qi in range(Sq):
            cmax = Sk - Sq + qi
            bias = np.where(np.arange(Sk) <= cmax, 0.0, -np.inf) + am[0, qi].astype(np.float64)
            qd, kd, vd = q[0, h, qi].astype(np.float64), k[0, 0].astype(np.float64), \
                v[0, 0].astype(np.float64)
            _close(got[0, h, qi], _stream_tiles(qd, kd, vd, bias, scale, 16), 1e-12,
                   f"tile recurrence h={h} qi={qi}")
            _close(got[0, h, qi], _stream_keys(qd, kd, vd, bias, scale), 1e-12,
                   f"per-key recurrence h={h} qi={qi}")


def pin_uniform_v(lib):
    rng = np.random.default_rng(13)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 6, 11, 5
    q, k = _rand(rng, B, Hq, Sq, D, std=3.0), _rand(rng, B, Hkv, Sk, D, std=3.0)
    row = _rand(rng, D)
    v = np.broadcast_to(row, (B, Hkv, Sk, D)).copy()
    for kw in ({}, {"causal": True}, {"causal": True, "local_window": 3}):
        got = _run(lib, q, k, v, **kw)
        _close(got, np.broadcast_to(row, got.shape), 1e-13, f"uniform V {kw}")


def pin_mask_properties(lib):
    rng = np.random.default_rng(14)
    B, Hq, Hkv, Sq, Sk, D = 2, 2, 1, 4, 7, 6
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
    # mask values on a 1/256 grid and integer shifts, so the shifted mask is exact in f32
    am = (np.round(_rand(rng, B, Sq, Sk) * 256) / 256).astype(np.float32)
    base = _run(lib, q, k, v, mask=am, mask_planes=B)
    # a constant added to a whole mask row changes nothing
    shifted = am + rng.integers(-3, 4, size=(B, Sq, 1)).astype(np.float32)
    _close(_run(lib, q, k, v, mask=shifted, mask_planes=B), base, 1e-12, "mask row shift")
    # a -inf mask entry equals deleting that key
    j = 4
    am2 = am.copy()
    am2[:, :, j] = -np.inf
    keep = [x for x in range(Sk) if x != j]
    _close(_run(lib, q, k, v, mask=am2, mask_planes=B),
           _run(lib, q, k[:, :, keep], v[:, :, keep], mask=am[:, :, keep].copy(), mask_planes=B),
           1e-12, "-inf entry = deleted key")
    # rows masked entirely give 0
    am3 = am.copy()
    am3[1, 2, :] = -np.inf
    got = _run(lib, q, k, v, mask=am3, mask_planes=B)
    assert np.all(got[1, :, 2] == 0.0), "fully masked row is not 0"
    # shared plane (mask_planes = 1) equals the same plane given per batch and per head
    one = am[:1]
    ref = _run(lib, q, k, v, mask=one, mask_planes=1)
    _close(_run(lib, q, k, v, mask=np.repeat(one, B, 0), mask_planes=B), ref, 0.0,
           "per-batch copy of one plane")
    _close(_run(lib, q, k, v, mask=np.repeat(one, B * Hq, 0), mask_planes=B * Hq), ref, 0.0,
           "per-head copy of one plane")
    # per-batch planes equal per-head planes repeated over heads
    _close(_run(lib, q, k, v, mask=np.repeat(am, Hq, 0), mask_planes=B * Hq), base, 0.0,
           "per-head expansion of per-batch planes")


def pin_window_and_softcap_limits(lib):
    rng = np.random.default_rng(15)
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 6, 9, 4
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
    # window 1 with causal: each row copies V[causal_max] (causal_max = Sk - Sq + qi)
    got = _run(lib, q, k, v, causal=True, local_window=1)
    for h in range(Hq):
        for qi in range(Sq):
            _close(got[0, h, qi], v[0, h, Sk - Sq + qi], 0.0, f"window 1 row {qi}")
    # a window at least Sk wide equals no window
    _close(_run(lib, q, k, v, causal=True, local_window=Sk),
           _run(lib, q, k, v, causal=True), 0.0, "window >= Sk")
    _close(_run(lib, q, k, v, local_window=10 * Sk), _run(lib, q, k, v), 0.0, "huge window")
    # a huge soft-cap equals none; soft-cap with two keys has a closed form
    _close(_run(lib, q, k, v, softcap=1e30), _run(lib, q, k, v), 1e-12, "softcap 1e30")
    c, scale = 0.7, 0.9
    q2, k2, v2 = q[:, :, :1], k[:, :1, :2].copy(), v[:, :1, :2].copy()
    got = _run(lib, q2, k2, v2, softcap=c, scale=scale)
    for h in range(Hq):
        s = [c * math.tanh(scale * float(np.dot(q2[0, h, 0].astype(np.float64),
                                                k2[0, 0, j].astype(np.float64))) / c)
             for j in range(2)]
        w1 = 1.0 / (1.0 + math.exp(s[0] - s[1]))
        expect = (1 - w1) * v2[0, 0, 0].astype(np.float64) + w1 * v2[0, 0, 1].astype(np.float64)
        _close(got[0, h, 0], expect, 1e-13, "two-key soft-cap closed form")


def pin_gqa_and_layout(lib):
    rng = np.random.default_rng(16)
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 2, 5, 8, 4
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
    g = Hq // Hkv
    gqa = _run(lib, q, k, v, causal=True)
    mha = _run(lib, q, np.repeat(k, g, 1), np.repeat(v, g, 1), causal=True)
    _close(gqa, mha, 0.0, "GQA = MHA with replicated K/V")
    tok = _run(lib, q, k, v, causal=True, out_layout=1)
    _close(tok, gqa.transpose(0, 2, 1, 3).reshape(B, Sq, Hq * D), 0.0, "token-major transpose")


def pin_ragged(lib):
    rng = np.random.default_rng(17)
    B, Hq, Hkv, Sq, cap, D = 3, 4, 2, 4, 12, 4
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, cap, D), _rand(rng, B, Hkv, cap, D)
    # past = 0, total = Sq equals plain causal on the first Sq keys
    total = np.full(B, Sq, np.int32)
    past = np.zeros(B, np.int32)
    _close(_run(lib, q, k, v, causal=True, total=total, past=past),
           _run(lib, q, k[:, :, :Sq].copy(), v[:, :, :Sq].copy(), causal=True), 0.0,
           "ragged past=0 = plain causal")
    # ragged batch b equals a dense problem on K/V sliced to total[b]
    past = np.array([0, 3, 8], np.int32)
    total = past + Sq
    am = _rand(rng, B, Sq, cap)
    got = _run(lib, q, k, v, causal=True, total=total, past=past, mask=am, mask_planes=B)
    for b in range(B):
        t = int(total[b])
        dense = _run(lib, q[b:b + 1], k[b:b + 1, :, :t].copy(), v[b:b + 1, :, :t].copy(),
                     causal=True, mask=am[b:b + 1, :, :t].copy(), mask_planes=1)
        _close(got[b:b + 1], dense, 0.0, f"ragged batch {b} = sliced dense")
    # garbage (including NaN / inf) in slots >= total changes nothing
    k2, v2 = k.copy(), v.copy()
    for b in range(B):
        t = int(total[b])
        k2[b, :, t:] = np.nan
        v2[b, :, t:] = np.inf
    _close(_run(lib, q, k2, v2, causal=True, total=total, past=past, mask=am, mask_planes=B),
           got, 0.0, "garbage slots")
    # Sk < kv_capacity: slots in [Sk, cap) are never read
    k3, v3 = k.copy(), v.copy()
    k3[:, :, 9:] = np.nan
    v3[:, :, 9:] = np.nan
    _close(_run(lib, q, k3, v3, Sk=9, causal=True),
           _run(lib, q, k[:, :, :9].copy(), v[:, :, :9].copy(), causal=True), 0.0,
           "Sk < kv_capacity")
    # the mask row stride is Sk, not kv_capacity: the mask buffer is padded so a wrong
    # stride reads defined (wrong) values instead of running off the end
    am9 = _rand(rng, B, Sq, 9)
    padded = np.zeros(B * Sq * cap, dtype=np.float32)
    padded[:am9.size] = am9.ravel()
    _close(_run(lib, q, k, v, Sk=9, mask=padded, mask_planes=B),
           _run(lib, q, k[:, :, :9].copy(), v[:, :, :9].copy(), mask=am9, mask_planes=B),
           0.0, "mask stride Sk")


def pin_brute_force_tiny(lib):
    """Every shape up to 3x3 with D <= 3 against an explicit softmax built
    with scipy's softmax over the visible keys."""
    from scipy.special import softmax
    rng = np.random.default_rng(18)
    for Sq in (1, 2, 3):
        for Sk in (1, 2, 3):
            for D in (1, 2, 3):
                for causal in (False, True):
                    q, k, v = _rand(rng, 1, 1, Sq, D), _rand(rng, 1, 1, Sk, D), \
                        _rand(rng, 1, 1, Sk, D)
                    got = _run(lib, q, k, v, causal=causal, scale=0.8)
                    for qi in range(Sq):
                        keys = [j for j in range(Sk) if not causal or j <= Sk - Sq + qi]
                        if not keys:
                            _close(got[0, 0, qi], np.zeros(D), 0.0, "empty row")
                            continue
                        s = np.array([0.8 * float(np.dot(q[0, 0, qi].astype(np.float64),
                                                         k[0, 0, j].astype(np.float64)))
                                      for j in keys])
                        p = softmax(s)
                        expect = p @ v[0, 0, keys].astype(np.float64)
                        _close(got[0, 0, qi], expect, 1e-13, f"tiny {Sq}x{Sk}x{D} c={causal}")


def pin_rows_equal_full(lib):
    """oracle_attn_rows (rows one by one, any order) equals the full forward."""
    rng = np.random.default_rng(19)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 9, 13, 5
    q, k, v = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
    am = _rand(rng, B * Hq, Sq, Sk)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, kv_capacity=Sk, D=D, causal=True,
              local_window=5, scale=0.7, softcap=2.0, mask=am, mask_planes=B * Hq, nthreads=3,
              lib=lib)
    full = oracle.attn_fwd(q, k, v, **kw)
    rows = np.array([(b, h, i) for b in range(B) for h in range(Hq) for i in range(Sq)])[::-1]
    got = oracle.attn_rows(q, k, v, rows, **kw)
    _close(got, full[rows[:, 0], rows[:, 1], rows[:, 2]], 0.0, "rows = full")


def pin_lse(lib):
    """The row log-sum-exp: hand-worked values, scipy's logsumexp over the
    explicitly formed score rows, and the shift a constant mask row causes."""
    from scipy.special import logsumexp
    eye = np.eye(2, dtype=np.float32).reshape(1, 1, 2, 2)
    v = np.array([[1, 2], [3, 4]], np.float32).reshape(1, 1, 2, 2)
    kw = dict(B=1, Hq=1, Hkv=1, Sq=2, Sk=2, kv_capacity=2, D=2, scale=1.0, nthreads=1, lib=lib)
    _, lse = oracle.attn_fwd_lse(eye, eye, v, **kw)
    _close(lse[0, 0], [math.log(math.e + 1), math.log(1 + math.e)], 1e-14, "lse plain 2x2")
    _, lse = oracle.attn_fwd_lse(eye, eye, v, causal=True, **kw)
    _close(lse[0, 0], [1.0, math.log(1 + math.e)], 1e-14, "lse causal 2x2")
    m = np.array([[[-np.inf, -np.inf], [0, 0]]], np.float32)
    _, lse = oracle.attn_fwd_lse(eye, eye, v, mask=m, mask_planes=1, **kw)
    assert lse[0, 0, 0] == -np.inf, "fully masked row must have lse -inf"
    rng = np.random.default_rng(20)
    B, Hq, Hkv, Sq, Sk, D = 2, 4, 2, 7, 11, 6
    q, k, vv = _rand(rng, B, Hq, Sq, D), _rand(rng, B, Hkv, Sk, D), _rand(rng, B, Hkv, Sk, D)
    am = (np.round(_rand(rng, B, Sq, Sk) * 256) / 256).astype(np.float32)
    scale, c = 0.6, 3.0
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Sk=Sk, kv_capacity=Sk, D=D, scale=scale, causal=True,
              softcap=c, mask=am, mask_planes=B, nthreads=2, lib=lib)
    out, lse = oracle.attn_fwd_lse(q, k, vv, **kw)
    _close(out, _run(lib, q, k, vv, causal=True, scale=scale, softcap=c, mask=am, mask_planes=B),
           0.0, "attn_fwd_lse output = attn_fwd output")
    g = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            s = scale * (q[b, h].astype(np.float64) @ k[b, h // g].astype(np.float64).T)
            s = c * np.tanh(s / c) + am[b].astype(np.float64)
            s[np.triu(np.ones((Sq, Sk), bool), k=Sk - Sq + 1)] = -np.inf
            _close(lse[b, h], logsumexp(s, axis=1), 1e-12, f"lse vs scipy b={b} h={h}")
    shift = rng.integers(-3, 4, size=(B, Sq, 1)).astype(np.float32)
    _, lse2 = oracle.attn_fwd_lse(q, k, vv, **dict(kw, mask=am + shift))
    _close(lse2, lse + np.repeat(shift[:, None, :, 0], Hq, axis=1), 1e-12, "lse shift")


PINS = [pin_rows_equal_full, pin_lse, pin_closed_forms, pin_torch_sdpa, pin_streaming_recurrences, pin_uniform_v,
        pin_mask_properties, pin_window_and_softcap_limits, pin_gqa_and_layout, pin_ragged,
        pin_brute_force_tiny]
