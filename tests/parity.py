"""Helpers shared by the GPU parity tests: run a workload through the CUDA
library (C ABI via the binding) and through the fp64 oracle on the same
seeded inputs, and compare with the tolerances of the two kernel families.

Tolerances: the fp32 CUDA-core path must be within max-abs 1e-4 of the fp64
oracle; the bf16 / f16 tensor-core path within |got - exp| <= 2e-2 + 1e-2 |exp|
elementwise.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import tiled_online_softmax_02_gb300 as attn
from tiled_online_softmax_02_gb300.inputs import Workload, make_inputs

F32_ATOL = 1e-4
LP_ATOL, LP_RTOL = 2e-2, 1e-2


def to_dev(x: dict, dev="cuda") -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_gpu(w: Workload, x: dict, *, out=None):
    g = to_dev(x)
    o = attn.attn_fwd(g["q"], g["k"], g["v"], mask=g["mask"], total_lengths=g["total_lengths"],
                      past_lengths=g["past_lengths"], causal=w.causal,
                      local_window=w.local_window, scale=w.softmax_scale, softcap=w.softcap,
                      out_layout=w.out_layout, seq_k=w.Sk, out=out)
    torch.cuda.synchronize()
    st = attn.get_device_status()
    assert st == attn.ATTN_OK, f"device status {attn.status_string(st)}"
    return o


def run_gpu_f32split(w: Workload, x: dict, *, out=None, workspace=None):
    """The fp32 tensor-core entry (attn_fwd_f32_split) on the same inputs."""
    g = to_dev(x)
    o = attn.attn_fwd_f32_split(g["q"], g["k"], g["v"], mask=g["mask"],
                                total_lengths=g["total_lengths"], past_lengths=g["past_lengths"],
                                causal=w.causal, local_window=w.local_window,
                                scale=w.softmax_scale, softcap=w.softcap, out_layout=w.out_layout,
                                seq_k=w.Sk, out=out, workspace=workspace)
    torch.cuda.synchronize()
    st = attn.get_device_status()
    assert st == attn.ATTN_OK, f"device status {attn.status_string(st)}"
    return o


def run_oracle(w: Workload, x: dict):
    return oracle.attn_fwd(x["q"], x["k"], x["v"], B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk,
                           kv_capacity=w.kv_capacity, D=w.D, causal=w.causal,
                           local_window=w.local_window, scale=w.softmax_scale,
                           softcap=w.softcap, out_layout=w.out_layout, mask=x["mask"],
                           mask_planes=w.mask_planes, total_lengths=x["total_lengths"],
                           past_lengths=x["past_lengths"])


def oracle_rows(w: Workload, x: dict, rows: np.ndarray):
    return oracle.attn_rows(x["q"], x["k"], x["v"], rows, B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq,
                            Sk=w.Sk, kv_capacity=w.kv_capacity, D=w.D, causal=w.causal,
                            local_window=w.local_window, scale=w.softmax_scale,
                            softcap=w.softcap, mask=x["mask"], mask_planes=w.mask_planes,
                            total_lengths=x["total_lengths"], past_lengths=x["past_lengths"])


def gather_rows(w: Workload, out: torch.Tensor, rows: np.ndarray) -> np.ndarray:
    """Rows (b, h, qi) of the GPU output as float64 [n, D], either layout."""
    o = out
    if w.out_layout == 1:
        o = o.view(w.B, w.Sq, w.Hq, w.D).permute(0, 2, 1, 3)
    idx = torch.from_numpy(rows).to(o.device)
    sel = o[idx[:, 0], idx[:, 1], idx[:, 2]]
    return sel.double().cpu().numpy()


def check(w: Workload, got, ref, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    print(f"PARITY {what}: {got.size} elements, max abs err {float(err.max()) if err.size else 0.0:.3e}")
    if w.dtype == "f32":
        worst = float(err.max()) if err.size else 0.0
        assert worst <= F32_ATOL, f"{what}: f32 max abs err {worst:.3e} > {F32_ATOL}"
    else:
        bad = err > LP_ATOL + LP_RTOL * np.abs(ref)
        if bad.any():
            i = np.unravel_index(int(np.argmax(err - LP_RTOL * np.abs(ref))), err.shape)
            raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at "
                                 f"{i}: got {got[i]:.6f} expected {ref[i]:.6f}")
    return float(err.max()) if err.size else 0.0


def run_and_check(w: Workload, seed: int | None = None, what: str = ""):
    x = make_inputs(w, seed)
    out = run_gpu(w, x)
    ref = run_oracle(w, x)
    return check(w, out.double().cpu().numpy(), ref, what or w.name)


def run_oracle_lse(w: Workload, x: dict):
    return oracle.attn_fwd_lse(x["q"], x["k"], x["v"], B=w.B, Hq=w.Hq, Hkv=w.Hkv, Sq=w.Sq, Sk=w.Sk,
                               kv_capacity=w.kv_capacity, D=w.D, causal=w.causal,
                               local_window=w.local_window, scale=w.softmax_scale,
                               softcap=w.softcap, out_layout=w.out_layout, mask=x["mask"],
                               mask_planes=w.mask_planes, total_lengths=x["total_lengths"],
                               past_lengths=x["past_lengths"])


def run_gpu_splitkv(w: Workload, x: dict, num_splits: int):
    g = to_dev(x)
    o, lse = attn.attn_fwd_splitkv(g["q"], g["k"], g["v"], mask=g["mask"],
                                   total_lengths=g["total_lengths"], past_lengths=g["past_lengths"],
                                   causal=w.causal, local_window=w.local_window,
                                   scale=w.softmax_scale, softcap=w.softcap,
                                   out_layout=w.out_layout, seq_k=w.Sk, num_splits=num_splits)
    torch.cuda.synchronize()
    st = attn.get_device_status()
    assert st == attn.ATTN_OK, f"device status {attn.status_string(st)}"
    return o, lse


U_F32 = 2.0 ** -24          # unit roundoff of fp32
TANH_APPROX_REL = 2.0 ** -10  # tanh.approx.f32 relative error, with margin over its ~2^-11
EXP2_APPROX_REL = 2.0 ** -22  # ex2.approx / lg2.approx error


def lse_tolerance(w: Workload, x: dict) -> tuple[float, float]:
    """(atol, rtol) bounding |lse_gpu - lse_exact| for the 16-bit kernels' row
    log-sum-exp, derived from the fp32 arithmetic they do (u = 2^-24):

    - score: the tensor core adds D exact products of 16-bit values in fp32;
      each add errs by at most 2u of the running magnitude (2u also covers a
      truncating adder), so |ds| <= 2 D u A with A = max |scale| sum_d |q_d k_d|
      over the (row, key) pairs a row may see; scaling by scale log2 e and
      adding the mask round once more each: 2u (|s|max + |mask|max);
    - soft-cap: c tanh(s / c) through tanh.approx.f32 errs by its relative
      error times c |tanh(s / c)| <= min(|s|, c);
    - lse = log sum_j exp(s_j) moves by a p-weighted mean of the score errors,
      so by at most their maximum;
    - the exponentials (ex2.approx, relative 2^-22) and the row sum (at most
      Sk / 64 + 64 fp32 adds in sequence: sums inside a key tile, the running
      sum over tiles, the merge of split ranges) perturb l relatively, which
      is the same absolute error on log l;
    - the final lg2.approx (2^-22), the add m + log2 l and the change to the
      natural log: 2^-22 + 4u |lse|.

    A and the score maximum are taken over every key below each batch's
    valid length (a superset of the visible pairs), in fp64."""
    u = U_F32
    q = x["q"].detach().cpu().double()
    k = x["k"].detach().cpu().double()
    A = S = 0.0
    for b in range(w.B):
        lim = w.Sk
        if x.get("total_lengths") is not None:
            lim = min(lim, int(x["total_lengths"][b]))
        if lim <= 0:
            continue
        kb = k[b, :, :lim]                                   # [Hkv, lim, D]
        qb = q[b].reshape(w.Hkv, w.group * w.Sq, w.D)         # the heads of each kv head
        A = max(A, float((qb.abs() @ kb.abs().transpose(1, 2)).max()))
        S = max(S, float((qb @ kb.transpose(1, 2)).abs().max()))
    scale = abs(w.softmax_scale)
    A_s, S_s = scale * A, scale * S
    M = 0.0
    if x.get("mask") is not None:
        m = x["mask"].detach().cpu().double()
        fin = m[torch.isfinite(m)]
        M = float(fin.abs().max()) if fin.numel() else 0.0
    atol = 2 * w.D * u * A_s + 2 * u * (S_s + M)
    if w.softcap > 0:
        atol += TANH_APPROX_REL * min(S_s, w.softcap)
    atol += EXP2_APPROX_REL + (w.Sk / 64 + 64) * u + EXP2_APPROX_REL
    return atol, 4 * u


def check_lse(got, ref, what="", tol: tuple[float, float] | None = None):
    """Row log-sum-exps against the oracle's: rows without a finite score
    must be -inf on both sides; the rest within ``tol`` = (atol, rtol)
    (``lse_tolerance``).  Returns the largest error."""
    atol, rtol = tol if tol is not None else (LSE_ATOL_FALLBACK, 4 * U_F32)
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf rows differ"
    g, r = got[~both_inf], ref[~both_inf]
    assert np.isfinite(g).all(), f"{what}: non-finite lse"
    err = np.abs(g - r)
    worst = float(err.max()) if err.size else 0.0
    print(f"PARITY-LSE {what}: max err {worst:.3e}, tolerance {atol:.3e} + {rtol:.1e} |lse|")
    bad = err > atol + rtol * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} lse values out of tolerance " \
                          f"(max err {worst:.3e}, atol {atol:.3e})"
    return worst


# only for comparisons of two GPU results (no inputs at hand to derive a bound from)
LSE_ATOL_FALLBACK = 2e-4
