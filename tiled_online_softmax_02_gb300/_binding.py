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
    "attn_fwd_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp,
                             _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                             _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                             _i32, _i32, ctypes.c_float, ctypes.c_float, _i32,
                             _i32, _i32, _vp, _vp]),
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
_host_copies = threading.local()  # (h2d, d2h) bytes of this thread's last host-tensor call


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
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shape = (B, Hq, Sq, D) if layout == 0 else (B, Sq, Hq * D)
    if out is not None and (tuple(out.shape) != shape or out.dtype != q.dtype or not out.is_contiguous()):
        raise ValueError(f"out must be a contiguous {q.dtype} tensor of shape {shape}")
    lib = load_library()
    what = "attn_fwd_f32_split" if _f32_split else "attn_fwd"

    def launch(dq, dk, dv, dmask, dtot, dpast, dout, b_, hq_, hkv_, planes, ws, stream):
        args = (_ptr(dq), _ptr(dk), _ptr(dv), _ptr(dmask), _ptr(dtot), _ptr(dpast), _ptr(dout), b_, hq_, hkv_,
                Sq, Sk, kv_capacity, D, int(bool(causal)), int(local_window), float(scale), float(softcap),
                layout, planes)
        if _f32_split:
            ws_bytes = ws.numel() * ws.element_size()
            return lib.attn_fwd_f32_split(*args, _ptr(ws), ws_bytes, stream)
        return lib.attn_fwd(*args, DTYPE_CODES[q.dtype], stream)

    if not q.is_cuda:
        return _host_pipeline(q, k, v, mask, total_lengths, past_lengths, out, shape, layout, mask_planes,
                              launch, lib, _f32_split, what,
                              (Sk, int(bool(causal)), int(local_window), float(scale), float(softcap)))
    if out is None:
        out = torch.empty(shape, dtype=q.dtype, device=q.device)
    with torch.cuda.device(q.device):
        ws = None
        if _f32_split:
            need = lib.attn_f32_split_workspace_bytes(B, Hkv, kv_capacity, D)
            ws = workspace if (workspace is not None and workspace.is_cuda) else \
                torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        rc = launch(q, k, v, mask, total_lengths, past_lengths, out, B, Hq, Hkv, mask_planes, ws,
                    _stream_handle(q.device))
    if rc != ATTN_OK:
        raise AttnError(rc, what)
    return out


def host_copy_bytes():
    """(host-to-device, device-to-host) bytes the calling thread's last
    attention call on host tensors copied; (0, 0) before the first."""
    return getattr(_host_copies, "value", (0, 0))


def _host_pieces(B, Hq, Hkv, layout):
    """The host path's pieces of a problem, (b0, b1, h0, h1, kv0, kv1): runs
    of whole batches, at most 64 pieces, and -- for head-major output, whose
    head slices are contiguous -- with fewer than eight batches each batch
    cut further by whole kv-head groups, so that about eight pieces exist to
    overlap with one another.  attn_fwd_host cuts by the same rule."""
    group = Hq // Hkv
    pieces = []
    if layout == 0 and B < 8:
        per_batch = min(Hkv, -(-8 // max(B, 1)))
        for b in range(B):
            for i in range(per_batch):
                kv0, kv1 = Hkv * i // per_batch, Hkv * (i + 1) // per_batch
                if kv1 > kv0:
                    pieces.append((b, b + 1, kv0 * group, kv1 * group, kv0, kv1))
        return pieces
    chunks = min(B, 64)
    for i in range(chunks):
        b0, b1 = B * i // chunks, B * (i + 1) // chunks
        if b1 > b0:
            pieces.append((b0, b1, 0, Hq, 0, Hkv))
    return pieces


def _host_pipeline(q, k, v, mask, total_lengths, past_lengths, host_out, shape, layout, mask_planes, launch,
                   lib, f32_split, what, params):
    """The end-to-end path for host (ideally pinned) tensors.  The problem is
    cut into contiguous pieces (_host_pieces), each an ordinary call on its
    slices, and three streams overlap piece i + 1's upload, piece i's kernel
    and piece i - 1's download.  Every piece computes exactly what the whole
    call would for its rows, so the result is the same bit for bit.  For
    attn_fwd the library issues the pipeline itself (_host_native); the fp32
    split path issues it from here."""
    B, Hq, Sq, D = q.shape
    Hkv, kv_capacity = k.shape[1], k.shape[2]
    dev = torch.device("cuda", torch.cuda.current_device())
    if host_out is None:
        host_out = torch.empty(shape, dtype=q.dtype, pin_memory=True)
    if not f32_split:
        return _host_native(q, k, v, mask, total_lengths, past_lengths, host_out, layout, mask_planes, lib, dev,
                            params)
    with torch.cuda.device(dev):
        compute = torch.cuda.current_stream(dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_in.wait_stream(compute)  # device buffers may be reused from earlier work on this stream
        dq, dk, dv = (torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q, k, v))
        dout = torch.empty(shape, dtype=q.dtype, device=dev)
        dtot = None if total_lengths is None else torch.empty_like(total_lengths, device=dev)
        dpast = None if past_lengths is None else torch.empty_like(past_lengths, device=dev)
        dmask = None if mask is None else torch.empty(mask.shape, dtype=mask.dtype, device=dev)
        pieces = _host_pieces(B, Hq, Hkv, layout) if B > 0 and Sq > 0 else []
        ws = None
        if f32_split and pieces:
            need = max(lib.attn_f32_split_workspace_bytes(b1 - b0, kv1 - kv0, kv_capacity, D)
                       for b0, b1, _, _, kv0, kv1 in pieces)
            ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        up = down = 0
        with torch.cuda.stream(s_in):
            for src, dst in ((total_lengths, dtot), (past_lengths, dpast)):
                if src is not None:
                    dst.copy_(src, non_blocking=True)
                    up += src.numel() * 4
            if mask is not None and mask_planes == 1:
                up += mask.numel() * 4
                dmask.copy_(mask, non_blocking=True)  # one plane shared by every piece
        mask_batch = -1  # batch whose plane was last uploaded (per-batch planes)
        for b0, b1, h0, h1, kv0, kv1 in pieces:
            nb, hq_, hkv_ = b1 - b0, h1 - h0, kv1 - kv0
            planes = 0
            m_host = m_dev = None
            if mask is not None:
                if mask_planes == 1:
                    m_dev, planes = dmask, 1
                elif mask_planes == B and not (mask_planes == B * Hq and Hq > 1):
                    m_dev, planes = dmask[b0:b1], nb
                    if b0 != mask_batch:  # a batch's plane goes up once, with its first piece
                        m_host, mask_batch = mask[b0:b1], b0
                else:  # a plane per (batch, head); the piece's planes are contiguous
                    p0, p1 = b0 * Hq + h0, (b1 - 1) * Hq + h1
                    m_host, m_dev, planes = mask[p0:p1], dmask[p0:p1], p1 - p0
            slices_h = (q[b0:b1, h0:h1], k[b0:b1, kv0:kv1], v[b0:b1, kv0:kv1])
            slices_d = (dq[b0:b1, h0:h1], dk[b0:b1, kv0:kv1], dv[b0:b1, kv0:kv1])
            o_d = dout[b0:b1, h0:h1] if layout == 0 else dout[b0:b1]
            o_h = host_out[b0:b1, h0:h1] if layout == 0 else host_out[b0:b1]
            with torch.cuda.stream(s_in):
                for src, dst in zip(slices_h, slices_d):
                    dst.copy_(src, non_blocking=True)
                    up += src.numel() * src.element_size()
                if m_host is not None:
                    m_dev.copy_(m_host, non_blocking=True)
                    up += m_host.numel() * 4
                uploaded = torch.cuda.Event()
                uploaded.record(s_in)
            compute.wait_event(uploaded)
            rc = launch(*slices_d, m_dev, None if dtot is None else dtot[b0:b1],
                        None if dpast is None else dpast[b0:b1], o_d, nb, hq_, hkv_, planes, ws,
                        ctypes.c_void_p(compute.cuda_stream))
            if rc != ATTN_OK:
                compute.synchronize()
                raise AttnError(rc, what)
            computed = torch.cuda.Event()
            computed.record(compute)
            s_out.wait_event(computed)
            with torch.cuda.stream(s_out):
                o_h.copy_(o_d, non_blocking=True)
                down += o_h.numel() * o_h.element_size()
        s_out.synchronize()
        compute.wait_stream(s_out)
    _host_copies.value = (up, down)
    return host_out


def _host_native(q, k, v, mask, total_lengths, past_lengths, host_out, layout, mask_planes, lib, dev, params):
    """attn_fwd on host tensors through attn_fwd_host: one blocking library
    call that pipelines the pieces on the library's own streams.  The device
    copies of every argument are carved from one allocation."""
    B, Hq, Sq, D = q.shape
    Hkv, kv_capacity = k.shape[1], k.shape[2]
    args = (q, k, v, mask, total_lengths, past_lengths, host_out)
    sizes = [0 if t is None else t.numel() * t.element_size() for t in args]
    offsets, total = [], 0
    for n in sizes:
        offsets.append(total)
        total += -(-n // 256) * 256
    copied = (ctypes.c_uint64 * 2)()
    with torch.cuda.device(dev):
        buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
        base = buf.data_ptr()
        dptr = [None if t is None else ctypes.c_void_p(base + o) for t, o in zip(args, offsets)]
        rc = lib.attn_fwd_host(*(_ptr(t) for t in args), *dptr, B, Hq, Hkv, Sq, params[0], kv_capacity, D,
                               *params[1:], layout, mask_planes, DTYPE_CODES[q.dtype], _stream_handle(dev), copied)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_host")
    _host_copies.value = (int(copied[0]), int(copied[1]))
    return host_out


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
