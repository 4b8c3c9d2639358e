"""Seeded synthetic workloads for attention forward.

This module only describes problem shapes and draws seeded random inputs.  It
holds none of the attention arithmetic, so both the CUDA path (tests, bench)
and the CPU oracle can consume what it produces without sharing any method
code.  Values are drawn in float32 and then rounded to the workload's dtype;
both sides consume the rounded values (the oracle reads them widened to
float32, which holds every bf16 / f16 value exactly).

The shapes follow the two attention pages: the prefill / KV-cache kernel of
"onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs" (grouped
query heads, causal, window, soft-cap, additive mask, ragged lengths over a
kv_capacity-strided cache) and the DiT joint attention of "pictor-kernels
0.1.0, src/gpu_backend/cuda_imagen_attn_kernels.rs" (24 heads, seq 1536,
head_dim 128, non-causal, token-major output).  No public dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np
import torch

SEED_BASE = 0xA77E0000

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    kv_capacity: int
    D: int
    dtype: str                      # "f32" | "bf16" | "f16"
    causal: bool
    local_window: int = 0
    softcap: float = 0.0
    out_layout: int = 0             # 0 head-major [B,Hq,Sq,D]; 1 token-major [B,Sq,Hq*D]
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    mask: str | None = None         # None | "per_batch" | "per_head" | "shared"
    mask_neg_inf_frac: float = 0.0
    ragged: bool = False            # past ~ U{0..Sk-Sq}, total = past + Sq
    past_max: int | None = None     # override of the ragged past upper bound
    garbage: str | None = None      # None | "finite" | "nonfinite" (slots >= total)
    seed: int = SEED_BASE
    scale: float | None = None      # None -> 1/sqrt(D)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def mask_planes(self) -> int:
        if self.mask is None:
            return 0
        return {"per_batch": self.B, "per_head": self.B * self.Hq, "shared": 1}[self.mask]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads, in order; seed = SEED_BASE + index.
WORKLOADS: dict[str, Workload] = {}


def _add(idx: int, w: Workload) -> None:
    WORKLOADS[w.name] = w.replace(seed=SEED_BASE + idx)


_add(0, Workload("tiny_f32", B=1, Hq=2, Hkv=1, Sq=64, Sk=64, kv_capacity=64, D=64,
                 dtype="f32", causal=True))
_add(1, Workload("dit_f32", B=1, Hq=24, Hkv=24, Sq=1536, Sk=1536, kv_capacity=1536, D=128,
                 dtype="f32", causal=False, out_layout=1))
_add(2, Workload("gqa_causal_bf16", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, kv_capacity=4096,
                 D=128, dtype="bf16", causal=True))
_add(3, Workload("window_softcap_bf16", B=4, Hq=16, Hkv=8, Sq=8192, Sk=8192,
                 kv_capacity=8192, D=128, dtype="bf16", causal=True, local_window=1024,
                 softcap=50.0, q_std=math.sqrt(2.0), k_std=math.sqrt(2.0)))
_add(4, Workload("ragged_kvcache_f16", B=8, Hq=32, Hkv=4, Sq=128, Sk=4096, kv_capacity=4096,
                 D=128, dtype="f16", causal=True, mask="per_batch", mask_neg_inf_frac=0.1,
                 ragged=True, garbage="finite"))

WORKLOAD_ORDER = list(WORKLOADS)

# Shapes beyond the five: decode (one new token per sequence over a long
# ragged cache), the case split-KV serves; and the wider head dims of the DiT
# page's kernel variants (256 and 384).
EXTRA_WORKLOADS: dict[str, Workload] = {
    "decode_bf16": Workload("decode_bf16", B=8, Hq=32, Hkv=8, Sq=1, Sk=32768, kv_capacity=32768,
                            D=128, dtype="bf16", causal=True, ragged=True, garbage="finite",
                            seed=SEED_BASE + 10),
    "gqa_causal_bf16_d256": Workload("gqa_causal_bf16_d256", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096,
                                     kv_capacity=4096, D=256, dtype="bf16", causal=True,
                                     seed=SEED_BASE + 11),
    # the widest head dim of the DiT page's kernel variants (384, its VAE
    # variant): the same GQA causal prefill in bf16, and an fp32 VAE-style
    # attention (non-causal, token-major output, as the page's op) over a
    # 32 x 32 latent grid
    "gqa_causal_bf16_d384": Workload("gqa_causal_bf16_d384", B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096,
                                     kv_capacity=4096, D=384, dtype="bf16", causal=True,
                                     seed=SEED_BASE + 12),
    "vae_f32_d384": Workload("vae_f32_d384", B=1, Hq=4, Hkv=4, Sq=1024, Sk=1024, kv_capacity=1024,
                             D=384, dtype="f32", causal=False, out_layout=1, seed=SEED_BASE + 13),
}


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(TORCH_DTYPES[dtype])


def make_lengths(w: Workload, rng: np.random.Generator):
    """Ragged lengths: past ~ U{0..past_max} inclusive, total = past + Sq."""
    if not w.ragged:
        return None, None
    hi = w.past_max if w.past_max is not None else w.Sk - w.Sq
    past = rng.integers(0, hi + 1, size=w.B, dtype=np.int64)
    total = past + w.Sq
    return (torch.from_numpy(total.astype(np.int32)), torch.from_numpy(past.astype(np.int32)))


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Draw the workload's inputs on the CPU.

    Returns a dict with q [B,Hq,Sq,D], k / v [B,Hkv,kv_capacity,D] in the
    workload dtype, mask (f32 [planes,Sq,Sk] or None), total_lengths / past_lengths
    (int32 [B] or None).  Cache slots at or beyond total_lengths[b] (and beyond
    Sk) hold garbage when ``w.garbage`` is set, otherwise zeros.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    q = rng.standard_normal((w.B, w.Hq, w.Sq, w.D), dtype=np.float32) * np.float32(w.q_std)
    k = rng.standard_normal((w.B, w.Hkv, w.kv_capacity, w.D), dtype=np.float32) * np.float32(w.k_std)
    v = rng.standard_normal((w.B, w.Hkv, w.kv_capacity, w.D), dtype=np.float32) * np.float32(w.v_std)
    total, past = make_lengths(w, rng)

    # slots that no key index may read as valid data
    for b in range(w.B):
        lim = int(total[b]) if total is not None else w.Sk
        lim = max(0, min(lim, w.kv_capacity))
        n = w.kv_capacity - lim
        if n <= 0:
            continue
        if w.garbage == "finite":
            k[b, :, lim:, :] = rng.uniform(-1000.0, 1000.0, size=(w.Hkv, n, w.D)).astype(np.float32)
            v[b, :, lim:, :] = rng.uniform(-1000.0, 1000.0, size=(w.Hkv, n, w.D)).astype(np.float32)
        elif w.garbage == "nonfinite":
            pat = np.array([np.nan, np.inf, -np.inf, 3.0e4], dtype=np.float32)
            k[b, :, lim:, :] = pat[rng.integers(0, 4, size=(w.Hkv, n, w.D))]
            v[b, :, lim:, :] = pat[rng.integers(0, 4, size=(w.Hkv, n, w.D))]
        else:
            k[b, :, lim:, :] = 0.0
            v[b, :, lim:, :] = 0.0

    mask = None
    if w.mask is not None:
        m = rng.standard_normal((w.mask_planes, w.Sq, w.Sk), dtype=np.float32)
        if w.mask_neg_inf_frac > 0:
            m[rng.random((w.mask_planes, w.Sq, w.Sk)) < w.mask_neg_inf_frac] = -np.inf
        mask = torch.from_numpy(m)

    return dict(q=_round(q, w.dtype), k=_round(k, w.dtype), v=_round(v, w.dtype), mask=mask,
                total_lengths=total, past_lengths=past)


def sample_rows(w: Workload, n: int, seed: int = 7) -> np.ndarray:
    """A spread of (b, h, qi) rows: the first and last rows of every tile edge
    that matters plus seeded random rows.  Used to check full-size outputs on
    rows the oracle computes one by one."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = min(n, w.B * w.Hq * w.Sq)  # never ask for more rows than exist
    picks = set()
    for b in {0, w.B - 1}:
        for h in {0, w.Hq - 1, min(w.group, w.Hq - 1)}:
            for qi in {0, 1, 127, 128, w.Sq // 2, w.Sq - 129, w.Sq - 2, w.Sq - 1}:
                if 0 <= qi < w.Sq:
                    picks.add((b, h, qi))
    while len(picks) < n:
        picks.add((int(rng.integers(0, w.B)), int(rng.integers(0, w.Hq)),
                   int(rng.integers(0, w.Sq))))
    return np.array(sorted(picks), dtype=np.int64)


# ---------------------------------------------------------------------------
# DSA indexer index selection ("onnx-runtime-ep-cuda 0.1.0-dev.6,
# src/kernels/dsa_index_select.rs"): query [B, S, H, D], key [B, T, D],
# weights [B, S, H], bias f32 [B, 1, S, T].  The page gives no workload sizes;
# the synthetic ones below follow its use -- an indexer over a prefill (causal
# bias) and over decode steps with ragged cache lengths.
@dataclass(frozen=True)
class DsaWorkload:
    name: str
    B: int
    S: int
    H: int
    D: int
    T: int
    top_k: int
    dtype: str                      # "f32" | "bf16" | "f16"
    bias: str = "causal"            # "causal" | "causal_min" | "ragged_causal" | "random" | "zeros"
    weights_scale: float = 1.0
    q_std: float = 1.0
    k_std: float = 1.0
    w_std: float = 1.0
    ties: bool = False              # duplicate some key rows (exactly tied scores)
    seed: int = SEED_BASE + 20
    scale: float | None = None      # None -> 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def replace(self, **kw) -> "DsaWorkload":
        return dataclasses.replace(self, **kw)


DSA_WORKLOADS: dict[str, DsaWorkload] = {
    "dsa_prefill_bf16": DsaWorkload("dsa_prefill_bf16", B=1, S=4096, H=32, D=128, T=4096,
                                    top_k=2048, dtype="bf16", bias="causal", seed=SEED_BASE + 20),
    "dsa_decode_bf16": DsaWorkload("dsa_decode_bf16", B=8, S=1, H=32, D=128, T=32768, top_k=2048,
                                   dtype="bf16", bias="ragged_causal", seed=SEED_BASE + 21),
}


def make_dsa_inputs(w: DsaWorkload, seed: int | None = None) -> dict:
    """Seeded inputs of a DSA workload on the CPU: query / key / weights in the
    workload dtype, bias float32 [B, 1, S, T].  Bias modes: "causal" (0 on keys
    t <= T - S + s, -inf above), "causal_min" (the same with the most negative
    f32 as the fill), "ragged_causal" (per-batch valid length L_b ~ U{T/4..T},
    causal against its end, -inf beyond), "random" (N(0, 1) with 10% -inf),
    "zeros"."""
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    q = rng.standard_normal((w.B, w.S, w.H, w.D), dtype=np.float32) * np.float32(w.q_std)
    k = rng.standard_normal((w.B, w.T, w.D), dtype=np.float32) * np.float32(w.k_std)
    wt = rng.standard_normal((w.B, w.S, w.H), dtype=np.float32) * np.float32(w.w_std)
    if w.ties and w.T >= 4:
        # every fourth key repeats the key before it: those pairs tie exactly
        k[:, 3::4, :] = k[:, 2:-1:4, :][:, : k[:, 3::4, :].shape[1], :]
    s_idx = np.arange(w.S)[:, None]
    t_idx = np.arange(w.T)[None, :]
    bias = np.zeros((w.B, 1, w.S, w.T), dtype=np.float32)
    lengths = None
    if w.bias in ("causal", "causal_min"):
        fill = -np.inf if w.bias == "causal" else np.finfo(np.float32).min
        bias[:, 0] = np.where(t_idx <= (w.T - w.S) + s_idx, 0.0, fill)
    elif w.bias == "ragged_causal":
        lengths = rng.integers(max(1, w.T // 4), w.T + 1, size=w.B)
        for b in range(w.B):
            bias[b, 0] = np.where(t_idx <= (int(lengths[b]) - w.S) + s_idx, 0.0, -np.inf)
    elif w.bias == "random":
        bias[:] = rng.standard_normal(bias.shape, dtype=np.float32)
        bias[rng.random(bias.shape) < 0.1] = -np.inf
    elif w.bias != "zeros":
        raise ValueError(f"unknown bias mode {w.bias!r}")
    return dict(query=_round(q, w.dtype), key=_round(k, w.dtype), weights=_round(wt, w.dtype),
                bias=torch.from_numpy(bias), lengths=lengths)
