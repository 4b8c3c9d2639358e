"""Thin ctypes binding over libattn.so (include/attn.h).

Argument marshalling only: shapes are read off the tensors, the output is
allocated with torch when the caller passes none, and the call goes to the C
ABI on torch's current CUDA stream.  Every step of attention runs in the
library's CUDA kernels; there is no fallback of any kind, and a missing
library raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
DTYPE_CODES = {torch.float32: ATTN_F32, torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16}
LAYOUTS = {"head": 0, "head_major": 0, 0: 0, "token": 1, "token_major": 1, 1: 1}

# Every function include/attn.h declares, with its ctypes signature.
_vp, _i32, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
SIGNATURES = {
    "attn_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                        _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                        _i32, _i32, ctypes.c_float, ctypes.c_float, _i32,
                        _i32, _i32, _vp]),
    "attn_fwd_splitkv": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                _i32, _i32, ctypes.c_float, ctypes.c_float, _i32,
                                _i32, _i32, _i32, _vp, _vp, ctypes.c_size_t, _vp]),
    "attn_fwd_splitkv_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                        _i32, _i32, ctypes.c_float, ctypes.c_float, _i32,
                                        _i32, _i32, _i32, _vp, _vp]),
    "attn_fwd_f32_split": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                  _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                  _i32, _i32, ctypes.c_float, ctypes.c_float, _i32,
                                  _i32, _vp, ctypes.c_size_t, _vp]),
    "attn_f32_split_workspace_bytes": (ctypes.c_size_t, [_i32, _i32, _i32, _i32]),
    "dsa_index_select": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                ctypes.c_float, ctypes.c_float, _i32, _vp, ctypes.c_size_t, _vp]),
    "dsa_index_select_workspace_bytes": (ctypes.c_size_t, [_i32, _i32, _i32]),
    "attn_splitkv_num_splits": (_i32, [_i32, _i32, _i32, _i32, _i32]),
    "attn_splitkv_workspace_bytes": (ctypes.c_size_t, [_i32, _i32, _i32, _i32, _i32]),
    "attn_status_string": (ctypes.c_char_p, [_i32]),
    "attn_last_cuda_error": (_i32, []),
    "attn_get_device_status": (_i32, [_vp]),
    "attn_set_wait_timeout_ns": (_i32, [_u64]),
    "attn_selftest_bounded_wait": (_i32, [_u64, _vp]),
    "attn_version": (_i32, []),
}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def library_path() -> str:
    """The in-tree libattn.so, or the file GB300_ATTN_LIBRARY names."""
    return os.environ.get("GB300_ATTN_LIBRARY") or _build.LIB


def load_library():
    """Load libattn.so; raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def attn_fwd(q, k, v, *, mask=None, total_lengths=None, past_lengths=None, causal=False,
             local_window=0, scale=None, softcap=0.0, out_layout="head", seq_k=None, out=None,
             _f32_split=False, workspace=None):
    """Attention forward through libattn.so.

    q [B, Hq, Sq, D]; k, v [B, Hkv, kv_capacity, D] (same dtype: float32,
    float16 or bfloat16); mask None or float32 [planes, Sq, Sk] (planes 1, B or
    B*Hq; a 4-D [B, Hq, Sq, Sk] or [B, 1, Sq, Sk] mask is viewed as such);
    total_lengths / past_lengths None or int32 [B]; seq_k = Sk (defaults to
    kv_capacity).  out_layout "head" -> [B, Hq, Sq, D], "token" ->
    [B, Sq, Hq*D].  scale defaults to 1/sqrt(D).

    CUDA tensors: the call is enqueued on torch's current stream and returns
    at once.  CPU tensors (ideally pinned): they are copied to the current
    CUDA device, the kernel runs, and the output is copied back into a CPU
    tensor (the end-to-end path).
    """
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D: [B, H, S, D]")
    B, Hq, Sq, D = q.shape
    Hkv, kv_capacity = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if q.dtype not in DTYPE_CODES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype among float32 / float16 / bfloat16")
    Sk = kv_capacity if seq_k is None else int(seq_k)
    layout = LAYOUTS[out_layout]
    mask_planes = 0
    if mask is not None:
        if mask.dtype != torch.float32:
            raise ValueError("mask must be float32")
        if mask.dim() == 4:
            mask = mask.reshape(-1, mask.shape[-2], mask.shape[-1])
        if mask.dim() != 3:
            raise ValueError("mask must be [planes, Sq, Sk]")
        mask_planes = mask.shape[0]
    for name, t in (("total_lengths", total_lengths), ("past_lengths", past_lengths)):
        if t is not None and (t.dtype != torch.int32 or t.numel() != B):
            raise ValueError(f"{name} must be int32 [B]")
    for t in (q, k, v, mask, total_lengths, past_lengths):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if t is not None and t.device != q.device:
            raise ValueError("all tensors must be on the same device")
    host = not q.is_cuda
    host_out = None
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())

        def up(t):
            return None if t is None else t.to(dev, non_blocking=True)
        q, k, v, mask, total_lengths, past_lengths = map(up, (q, k, v, mask, total_lengths,
                                                               past_lengths))
        host_out, out = out, None
    shape = (B, Hq, Sq, D) if layout == 0 else (B, Sq, Hq * D)
    if out is None:
        out = torch.empty(shape, dtype=q.dtype, device=q.device)
    elif tuple(out.shape) != shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous {q.dtype} tensor of shape {shape}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lib = load_library()
    with torch.cuda.device(q.device):
        args = (_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(total_lengths), _ptr(past_lengths),
                _ptr(out), B, Hq, Hkv, Sq, Sk, kv_capacity, D, int(bool(causal)),
                int(local_window), float(scale), float(softcap), layout, mask_planes)
        if _f32_split:
            need = lib.attn_f32_split_workspace_bytes(B, Hkv, kv_capacity, D)
            if workspace is None or not workspace.is_cuda:
                workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
            ws_bytes = workspace.numel() * workspace.element_size()
            rc = lib.attn_fwd_f32_split(*args, _ptr(workspace), ws_bytes, _stream_handle(q.device))
            what = "attn_fwd_f32_split"
        else:
            rc = lib.attn_fwd(*args, DTYPE_CODES[q.dtype], _stream_handle(q.device))
            what = "attn_fwd"
    if rc != ATTN_OK:
        raise AttnError(rc, what)
    if host:
        if host_out is None:
            host_out = torch.empty(shape, dtype=q.dtype, pin_memory=True)
        host_out.copy_(out, non_blocking=True)
        torch.cuda.current_stream(q.device).synchronize()
        return host_out
    return out


def attn_fwd_f32_split(q, k, v, *, mask=None, total_lengths=None, past_lengths=None,
                       causal=False, local_window=0, scale=None, softcap=0.0, out_layout="head",
                       seq_k=None, out=None, workspace=None):
    """fp32 attention forward on the tensor cores (attn_fwd_f32_split in the C
    ABI): q, k, v float32 with D = 64 or 128, carried as bf16 pieces: Q K^T as
    six bf16 products of three-piece operands, P V as three products of
    two-piece operands.  Arguments and result as attn_fwd (CUDA or,
    end to end, CPU tensors).  The bf16 workspace for the split K / V
    (attn_f32_split_workspace_bytes) is allocated with torch when not given."""
    if q.dtype != torch.float32:
        raise ValueError("attn_fwd_f32_split takes float32 q, k, v")
    return attn_fwd(q, k, v, mask=mask, total_lengths=total_lengths, past_lengths=past_lengths,
                    causal=causal, local_window=local_window, scale=scale, softcap=softcap,
                    out_layout=out_layout, seq_k=seq_k, out=out, _f32_split=True,
                    workspace=workspace)


def attn_fwd_splitkv(q, k, v, *, mask=None, total_lengths=None, past_lengths=None, causal=False,
                     local_window=0, scale=None, softcap=0.0, out_layout="head", seq_k=None,
                     num_splits=0, out=None, lse=None, workspace=None):
    """Split-KV attention forward (CUDA tensors, bf16 / f16): the same output
    as attn_fwd, computed over `num_splits` key ranges and merged (0 = the
    library's choice).  Returns (out, lse) with lse float32 [B, Hq, Sq], the
    natural-log log-sum-exp of each row's scores.  The fp32 workspace is
    allocated with torch when not given."""
    B, Hq, Sq, D = q.shape
    Hkv, kv_capacity = k.shape[1], k.shape[2]
    Sk = kv_capacity if seq_k is None else int(seq_k)
    lib = load_library()
    layout = LAYOUTS[out_layout]
    shape = (B, Hq, Sq, D) if layout == 0 else (B, Sq, Hq * D)
    if q.dtype not in (torch.float16, torch.bfloat16) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("split-KV needs float16 or bfloat16 q, k, v of one dtype")
    for t in (q, k, v, mask, total_lengths, past_lengths):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("split-KV takes contiguous CUDA tensors")
    mask_planes = 0
    if mask is not None:
        if mask.dim() == 4:
            mask = mask.reshape(-1, mask.shape[-2], mask.shape[-1])
        mask_planes = mask.shape[0]
    with torch.cuda.device(q.device):
        splits = int(num_splits) or lib.attn_splitkv_num_splits(B, Hq, Hkv, Sq, max(Sk, 1))
        need = lib.attn_splitkv_workspace_bytes(B, Hq, Sq, D, splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need // 4, dtype=torch.float32, device=q.device)
        if out is None:
            out = torch.empty(shape, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        rc = lib.attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(total_lengths),
                                  _ptr(past_lengths), _ptr(out), B, Hq, Hkv, Sq, Sk, kv_capacity,
                                  D, int(bool(causal)), int(local_window),
                                  float(1.0 / math.sqrt(D) if scale is None else scale),
                                  float(softcap), layout, mask_planes, DTYPE_CODES[q.dtype], splits,
                                  _ptr(lse), _ptr(workspace), ws_bytes, _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_splitkv")
    return out, lse


def dsa_index_select(query, key, weights, bias, *, top_k, scale, weights_scale=1.0, out=None,
                     workspace=None):
    """Sparse index selection of the DSA indexer (dsa_index_select in the C ABI).

    query [B, S, H, D], key [B, T, D], weights [B, S, H] (one dtype among
    float32 / float16 / bfloat16), bias float32 [B, 1, S, T].  Returns int64
    [B, 1, S, top_k]: per (b, s) the allowed keys (bias > -1e30) with the
    largest scores, ascending, then -1s.  CUDA tensors run on torch's current
    stream; CPU tensors are copied in and the result copied back.  The fp32
    score workspace is allocated with torch when not given."""
    if query.dim() != 4 or key.dim() != 3 or weights.dim() != 3 or bias.dim() != 4:
        raise ValueError("query [B,S,H,D], key [B,T,D], weights [B,S,H], bias [B,1,S,T]")
    B, S, H, D = query.shape
    T = key.shape[1]
    if tuple(key.shape) != (B, T, D) or tuple(weights.shape) != (B, S, H) or \
            tuple(bias.shape) != (B, 1, S, T):
        raise ValueError(f"shape mismatch: query {tuple(query.shape)} key {tuple(key.shape)} "
                         f"weights {tuple(weights.shape)} bias {tuple(bias.shape)}")
    if query.dtype not in DTYPE_CODES or key.dtype != query.dtype or weights.dtype != query.dtype:
        raise ValueError("query, key and weights must share one dtype among float32 / float16 / bfloat16")
    if bias.dtype != torch.float32:
        raise ValueError("bias must be float32")
    for t in (query, key, weights, bias):
        if not t.is_contiguous() or t.device != query.device:
            raise ValueError("inputs must be contiguous and on one device")
    host = not query.is_cuda
    if host:
        dev = torch.device("cuda", torch.cuda.current_device())
        query, key, weights, bias = (t.to(dev, non_blocking=True) for t in (query, key, weights, bias))
    shape = (B, 1, S, int(top_k))
    dev_out = out if (out is not None and out.is_cuda and not host) else \
        torch.empty(shape, dtype=torch.int64, device=query.device)
    if tuple(dev_out.shape) != shape or dev_out.dtype != torch.int64 or not dev_out.is_contiguous():
        raise ValueError(f"out must be a contiguous int64 tensor of shape {shape}")
    lib = load_library()
    with torch.cuda.device(query.device):
        need = lib.dsa_index_select_workspace_bytes(B, S, T)
        if workspace is None or not workspace.is_cuda:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=query.device)
        ws_bytes = workspace.numel() * workspace.element_size()
        rc = lib.dsa_index_select(_ptr(query), _ptr(key), _ptr(weights), _ptr(bias), _ptr(dev_out),
                                  B, S, H, D, T, int(top_k), float(scale), float(weights_scale),
                                  DTYPE_CODES[query.dtype], _ptr(workspace), ws_bytes,
                                  _stream_handle(query.device))
    if rc != ATTN_OK:
        raise AttnError(rc, "dsa_index_select")
    if host:
        res = out if out is not None else torch.empty(shape, dtype=torch.int64, pin_memory=True)
        res.copy_(dev_out, non_blocking=True)
        torch.cuda.current_stream(query.device).synchronize()
        return res
    return dev_out


def get_device_status(device=None) -> int:
    """Synchronises the current stream and returns (and clears) the device
    status word: ATTN_OK or ATTN_ERR_TIMEOUT."""
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        return load_library().attn_get_device_status(_stream_handle(dev))


def set_wait_timeout_ns(ns: int) -> None:
    load_library().attn_set_wait_timeout_ns(int(ns))


def selftest_bounded_wait(timeout_ns: int, device=None) -> int:
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        return load_library().attn_selftest_bounded_wait(int(timeout_ns), _stream_handle(dev))
