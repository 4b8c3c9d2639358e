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


# log-sum-exp: fp32 scores and sums against fp64
LSE_ATOL, LSE_RTOL = 2e-3, 1e-4


def check_lse(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf rows differ"
    g, r = got[~both_inf], ref[~both_inf]
    assert np.isfinite(g).all(), f"{what}: non-finite lse"
    bad = np.abs(g - r) > LSE_ATOL + LSE_RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} lse values out of tolerance " \
                          f"(max err {float(np.abs(g - r).max()):.3e})"
