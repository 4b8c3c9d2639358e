"""CPU oracle of the DSA indexer's sparse index selection -- TEST
INFRASTRUCTURE ONLY (see ``dsa_oracle.c`` for the definition and the page it
follows).  Only ``tests/`` and the CPU legs of ``bench.py`` use it.

The C file is compiled with ``-ffp-contract=off``: the page fixes the score
arithmetic to fp32 with every multiply and add rounded separately, in a set
order, and the selected indices depend on those exact bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_dsa.so")
# fp32 exactly as written: no contraction into FMA, no excess precision
CFLAGS = ("-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wextra", "-ffp-contract=off",
          "-fno-fast-math")

_lock = threading.Lock()
_lib = None


def build(force: bool = False, extra_cflags: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile ``dsa_oracle.c``; ``extra_cflags`` / ``out_path`` build variants
    (mutation tests) next to the real library."""
    path = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(path), exist_ok=True)
    if not force and not extra_cflags and os.path.exists(path) and \
            os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, *extra_cflags, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, path)
    return path


def _bind(lib):
    f32p = ctypes.POINTER(ctypes.c_float)
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    f32 = ctypes.c_float
    lib.oracle_dsa_scores.restype = ctypes.c_int
    lib.oracle_dsa_scores.argtypes = [f32p, f32p, f32p, f32p, f32p, u8p, i64, i64, i64, i64, i64, f32, f32]
    lib.oracle_dsa_select.restype = ctypes.c_int
    lib.oracle_dsa_select.argtypes = [f32p, u8p, i64p, i64, i64, i64]
    lib.oracle_dsa_rows.restype = ctypes.c_int
    lib.oracle_dsa_rows.argtypes = [f32p, f32p, f32p, f32p, i64p, i64, i64p, i64, i64, i64, i64, i64, i64,
                                    f32, f32]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle; ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _f32(a):
    if hasattr(a, "detach"):
        a = a.detach().float().cpu().numpy()
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _threads(nthreads: int) -> int:
    return nthreads if nthreads > 0 else (os.cpu_count() or 1)


def _run_chunks(fn, n: int, nthreads: int) -> None:
    """fn(i0, i1) over about-equal chunks of range(n), in threads (each chunk
    is one call into the C library, which releases the GIL)."""
    nt = max(1, min(_threads(nthreads), n))
    bounds = [n * i // nt for i in range(nt + 1)]
    if nt == 1:
        fn(0, n)
        return
    with ThreadPoolExecutor(nt) as ex:
        for f in [ex.submit(fn, bounds[i], bounds[i + 1]) for i in range(nt) if bounds[i + 1] > bounds[i]]:
            f.result()


def scores(query, key, weights, bias, *, scale, weights_scale=1.0, nthreads=1, lib=None):
    """Scores and allowed flags: (float32 [B, S, T], uint8 [B, S, T]).
    query [B, S, H, D], key [B, T, D], weights [B, S, H], bias [B, 1, S, T].
    ``nthreads`` > 1 (0: every core) splits the query rows over threads;
    every cell is still computed by the same C routine."""
    lib = lib or load()
    qa, _ = _f32(query)
    ka, _ = _f32(key)
    wa, _ = _f32(weights)
    ba, _ = _f32(bias)
    B, S, H, D = qa.shape
    T = ka.shape[1]
    sc = np.zeros((B, S, T), dtype=np.float32)
    al = np.zeros((B, S, T), dtype=np.uint8)
    f32p = ctypes.POINTER(ctypes.c_float)

    def part(b, s0, s1):
        # contiguous views of batch b, rows [s0, s1)
        q_, k_, w_ = qa[b, s0:s1], ka[b], wa[b, s0:s1]
        b_, sc_, al_ = ba[b, 0, s0:s1], sc[b, s0:s1], al[b, s0:s1]
        rc = lib.oracle_dsa_scores(q_.ctypes.data_as(f32p), k_.ctypes.data_as(f32p), w_.ctypes.data_as(f32p),
                                   b_.ctypes.data_as(f32p), sc_.ctypes.data_as(f32p),
                                   al_.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), 1, s1 - s0, H, D, T,
                                   float(scale), float(weights_scale))
        if rc != 0:
            raise ValueError(f"oracle_dsa_scores failed with code {rc}")

    def rows_fn(i0, i1):  # flat rows [i0, i1) of B * S, cut at batch boundaries
        while i0 < i1:
            b, s0 = divmod(i0, S)
            s1 = min(S, s0 + (i1 - i0))
            part(b, s0, s1)
            i0 += s1 - s0

    if nthreads == 1:  # one call over every batch
        rc = lib.oracle_dsa_scores(qa.ctypes.data_as(f32p), ka.ctypes.data_as(f32p), wa.ctypes.data_as(f32p),
                                   ba.ctypes.data_as(f32p), sc.ctypes.data_as(f32p),
                                   al.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), B, S, H, D, T,
                                   float(scale), float(weights_scale))
        if rc != 0:
            raise ValueError(f"oracle_dsa_scores failed with code {rc}")
    elif B * S > 0:
        _run_chunks(rows_fn, B * S, nthreads)
    return sc, al


def select(sc, allowed, top_k, *, lib=None):
    """Indices int64 [..., top_k] from scores / allowed [..., T]."""
    lib = lib or load()
    s = np.ascontiguousarray(np.asarray(sc, dtype=np.float32))
    a = np.ascontiguousarray(np.asarray(allowed, dtype=np.uint8))
    T = s.shape[-1]
    rows = int(np.prod(s.shape[:-1])) if s.ndim > 1 else 1
    out = np.zeros(s.shape[:-1] + (top_k,), dtype=np.int64)
    rc = lib.oracle_dsa_select(s.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                               a.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                               out.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows, T, int(top_k))
    if rc != 0:
        raise ValueError(f"oracle_dsa_select failed with code {rc}")
    return out


def index_select(query, key, weights, bias, *, top_k, scale, weights_scale=1.0, lib=None):
    """The whole op: int64 [B, 1, S, top_k]."""
    sc, al = scores(query, key, weights, bias, scale=scale, weights_scale=weights_scale, lib=lib)
    B, S, T = sc.shape
    return select(sc, al, top_k, lib=lib).reshape(B, 1, S, top_k)


def rows(query, key, weights, bias, row_ids, *, top_k, scale, weights_scale=1.0, nthreads=1, lib=None):
    """The op for selected rows (row = b * S + s): int64 [n, top_k].
    ``nthreads`` > 1 (0: every core) splits the rows over threads."""
    lib = lib or load()
    qa, qp = _f32(query)
    ka, kp = _f32(key)
    wa, wp = _f32(weights)
    ba, bp = _f32(bias)
    B, S, H, D = qa.shape
    T = ka.shape[1]
    r = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64).reshape(-1))
    out = np.zeros((r.shape[0], top_k), dtype=np.int64)
    i64p = ctypes.POINTER(ctypes.c_int64)

    def part(i0, i1):
        rc = lib.oracle_dsa_rows(qp, kp, wp, bp, r[i0:i1].ctypes.data_as(i64p), i1 - i0,
                                 out[i0:i1].ctypes.data_as(i64p), B, S, H, D, T, int(top_k), float(scale),
                                 float(weights_scale))
        if rc != 0:
            raise ValueError(f"oracle_dsa_rows failed with code {rc}")

    _run_chunks(part, r.shape[0], nthreads)
    return out
