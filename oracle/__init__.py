"""fp64 CPU oracle for attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or runs it, and this
package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use and marshals numpy arrays into it.
See that file's header for the definition it implements and the passages of
"onnx-runtime-ep-cuda 0.1.0-dev.5, src/kernels/flash_attention.rs" and
"pictor-kernels 0.1.0, src/gpu_backend/cuda_imagen_attn_kernels.rs" it
follows.  ``oracle.dsa`` is the oracle of the DSA indexer's index selection
("onnx-runtime-ep-cuda 0.1.0-dev.6, src/kernels/dsa_index_select.rs").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, extra_cflags: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile ``attn_oracle.c`` into a shared library and return its path.

    ``extra_cflags`` / ``out_path`` exist so tests can build deliberately
    broken variants of the oracle (mutation tests) next to the real one.
    """
    path = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(path), exist_ok=True)
    if not force and not extra_cflags and os.path.exists(path) and \
            os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra",
           *extra_cflags, "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    if out_path is None and not extra_cflags:
        from . import dsa  # the DSA indexer oracle, a library of its own
        dsa.build(force=force)
    return path


def _bind(lib):
    f32p = ctypes.POINTER(ctypes.c_float)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [f32p, f32p, f32p, f32p, i32p, i32p, f64p,
                                    i64, i64, i64, i64, i64, i64, i64,
                                    ctypes.c_int, i64, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_int, i64, ctypes.c_int]
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = [f32p, f32p, f32p, f32p, i32p, i32p, i64p, i64, f64p,
                                     i64, i64, i64, i64, i64, i64, i64,
                                     ctypes.c_int, i64, ctypes.c_double, ctypes.c_double,
                                     i64, ctypes.c_int]
    lib.oracle_attn_fwd_lse.restype = ctypes.c_int
    lib.oracle_attn_fwd_lse.argtypes = [f32p, f32p, f32p, f32p, i32p, i32p, f64p, f64p,
                                        i64, i64, i64, i64, i64, i64, i64,
                                        ctypes.c_int, i64, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_int, i64, ctypes.c_int]
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def default_threads() -> int:
    return int(load().oracle_default_threads())


def _f32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _i32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _as_numpy(t):
    """Accept numpy arrays or CPU torch tensors (any float dtype) as float32."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach()
        if t.dtype.is_floating_point:
            t = t.float()
        return t.cpu().numpy()
    return np.asarray(t)


def attn_fwd(q, k, v, *, B, Hq, Hkv, Sq, Sk, kv_capacity, D, causal=False,
             local_window=0, scale=None, softcap=0.0, out_layout=0, mask=None,
             mask_planes=0, total_lengths=None, past_lengths=None, nthreads=0,
             lib=None):
    """Full forward in fp64.  Returns float64 [B,Hq,Sq,D] or [B,Sq,Hq*D]."""
    lib = lib or load()
    if scale is None:
        scale = 1.0 / float(np.sqrt(D))
    qa, qp = _f32(_as_numpy(q))
    ka, kp = _f32(_as_numpy(k))
    va, vp = _f32(_as_numpy(v))
    ma, mp = _f32(_as_numpy(mask))
    ta, tp = _i32(_as_numpy(total_lengths))
    pa, pp = _i32(_as_numpy(past_lengths))
    shape = (B, Hq, Sq, D) if out_layout == 0 else (B, Sq, Hq * D)
    out = np.zeros(shape, dtype=np.float64)
    rc = lib.oracle_attn_fwd(qp, kp, vp, mp, tp, pp,
                             out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                             B, Hq, Hkv, Sq, Sk, kv_capacity, D, int(bool(causal)),
                             int(local_window), float(scale), float(softcap), int(out_layout),
                             int(mask_planes), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed with code {rc}")
    return out


def attn_rows(q, k, v, rows, *, B, Hq, Hkv, Sq, Sk, kv_capacity, D, causal=False,
              local_window=0, scale=None, softcap=0.0, mask=None, mask_planes=0,
              total_lengths=None, past_lengths=None, nthreads=0, lib=None):
    """Selected output rows in fp64.  ``rows`` is an int array [n, 3] of
    (b, h, qi); returns float64 [n, D]."""
    lib = lib or load()
    if scale is None:
        scale = 1.0 / float(np.sqrt(D))
    qa, qp = _f32(_as_numpy(q))
    ka, kp = _f32(_as_numpy(k))
    va, vp = _f32(_as_numpy(v))
    ma, mp = _f32(_as_numpy(mask))
    ta, tp = _i32(_as_numpy(total_lengths))
    pa, pp = _i32(_as_numpy(past_lengths))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((r.shape[0], D), dtype=np.float64)
    rc = lib.oracle_attn_rows(qp, kp, vp, mp, tp, pp,
                              r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), r.shape[0],
                              out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                              B, Hq, Hkv, Sq, Sk, kv_capacity, D, int(bool(causal)),
                              int(local_window), float(scale), float(softcap),
                              int(mask_planes), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed with code {rc}")
    return out


def attn_fwd_lse(q, k, v, *, B, Hq, Hkv, Sq, Sk, kv_capacity, D, causal=False,
                 local_window=0, scale=None, softcap=0.0, out_layout=0, mask=None,
                 mask_planes=0, total_lengths=None, past_lengths=None, nthreads=0, lib=None):
    """Full forward in fp64 plus the per-row log-sum-exp of the scores
    (natural log, -inf for rows without a finite score).  Returns (out, lse)
    with lse float64 [B, Hq, Sq]."""
    lib = lib or load()
    if scale is None:
        scale = 1.0 / float(np.sqrt(D))
    qa, qp = _f32(_as_numpy(q))
    ka, kp = _f32(_as_numpy(k))
    va, vp = _f32(_as_numpy(v))
    ma, mp = _f32(_as_numpy(mask))
    ta, tp = _i32(_as_numpy(total_lengths))
    pa, pp = _i32(_as_numpy(past_lengths))
    shape = (B, Hq, Sq, D) if out_layout == 0 else (B, Sq, Hq * D)
    out = np.zeros(shape, dtype=np.float64)
    lse = np.zeros((B, Hq, Sq), dtype=np.float64)
    f64p = ctypes.POINTER(ctypes.c_double)
    rc = lib.oracle_attn_fwd_lse(qp, kp, vp, mp, tp, pp, out.ctypes.data_as(f64p),
                                 lse.ctypes.data_as(f64p), B, Hq, Hkv, Sq, Sk, kv_capacity, D,
                                 int(bool(causal)), int(local_window), float(scale),
                                 float(softcap), int(out_layout), int(mask_planes), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_lse failed with code {rc}")
    return out, lse
