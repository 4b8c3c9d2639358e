"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every function include/attn.h declares, and rejects every invalid
request with the documented status before any CUDA call or launch."""
import ctypes
import math
import os
import re

import pytest

import tiled_online_softmax_02_gb300 as attn
from tiled_online_softmax_02_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return attn.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:attn|dsa)_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "attn_fwd" in names and "attn_status_string" in names
    assert set(names) == set(_binding.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(attn.library_path())
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} not exported"


def test_status_strings_and_version(lib):
    for code, name in [(0, "ATTN_OK"), (1, "ATTN_ERR_INVALID_ARG"), (2, "ATTN_ERR_UNSUPPORTED"),
                       (3, "ATTN_ERR_CUDA"), (4, "ATTN_ERR_TIMEOUT")]:
        assert lib.attn_status_string(code).decode() == name
    assert lib.attn_status_string(99).decode() == "ATTN_UNKNOWN_STATUS"
    assert lib.attn_version() == 100
    assert lib.attn_last_cuda_error() == 0


# fake, 16-byte aligned, non-overlapping device addresses: validation never
# dereferences them, and every case below fails before any CUDA call
Q, K, V, OUT, MASK, TOT, PAST = (0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000,
                                 0x60000000, 0x70000000)
GOOD = dict(q=Q, k=K, v=V, mask=None, total=None, past=None, out=OUT, B=2, Hq=4, Hkv=2, Sq=200,
            Sk=200, cap=200, D=64, causal=1, window=0, scale=0.125, softcap=0.0, layout=0,
            planes=0, dtype=2)


def call(lib, **kw):
    a = dict(GOOD, **kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["mask"], a["total"], a["past"], a["out"],
                        a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["cap"], a["D"], a["causal"],
                        a["window"], a["scale"], a["softcap"], a["layout"], a["planes"],
                        a["dtype"], None)


INVALID = {
    "dtype": dict(dtype=3),
    "negative_B": dict(B=-1),
    "negative_Sq": dict(Sq=-1),
    "zero_Hq": dict(Hq=0),
    "zero_Hkv": dict(Hkv=0),
    "zero_D": dict(D=0),
    "Hq_not_multiple": dict(Hq=5, Hkv=2),
    "negative_Sk": dict(Sk=-1),
    "Sk_over_capacity": dict(Sk=201),
    "causal_flag": dict(causal=2),
    "layout": dict(layout=2),
    "nan_scale": dict(scale=math.nan),
    "inf_scale": dict(scale=math.inf),
    "nan_softcap": dict(softcap=math.nan),
    "mask_without_planes": dict(mask=MASK, planes=0),
    "planes_without_mask": dict(planes=2),
    "bad_plane_count": dict(mask=MASK, planes=3),
    "negative_planes": dict(mask=MASK, planes=-1),
    "null_q": dict(q=None),
    "null_k": dict(k=None),
    "null_v": dict(v=None),
    "null_out": dict(out=None),
    "out_overlaps_q": dict(out=Q + 64),
    "out_overlaps_k": dict(out=K),
    "out_overlaps_mask": dict(mask=MASK, planes=2, out=MASK + 16),
    "out_overlaps_total_lengths": dict(total=TOT, out=TOT - 64),
    "out_overlaps_past_lengths": dict(past=PAST, out=PAST),
    "grid_z_too_large": dict(B=70000, Hq=2, Hkv=2, Sq=1, D=64),
    "size_overflow": dict(B=65535, Hq=65535, Hkv=65535, Sq=2**31 - 1, Sk=1, cap=2**31 - 1),
}


@pytest.mark.parametrize("case", list(INVALID))
def test_invalid_arguments(lib, case):
    assert call(lib, **INVALID[case]) == attn.ATTN_ERR_INVALID_ARG


UNSUPPORTED = {
    "bf16_d96": dict(D=96),
    "f16_d320": dict(D=320, dtype=1),
    "f32_d385": dict(D=385, dtype=0),
    "f32_d448": dict(D=448, dtype=0),
    "bf16_d512": dict(D=512),
    "misaligned_q": dict(q=Q + 8),
    "misaligned_out": dict(out=OUT + 2),
    "misaligned_mask": dict(mask=MASK + 2, planes=2),
    "misaligned_lengths": dict(total=TOT + 2),
}


@pytest.mark.parametrize("case", list(UNSUPPORTED))
def test_unsupported_requests(lib, case):
    assert call(lib, **UNSUPPORTED[case]) == attn.ATTN_ERR_UNSUPPORTED


def call_splitkv(lib, splits, ws=None, ws_bytes=0, lse=None, **kw):
    a = dict(GOOD, **kw)
    return lib.attn_fwd_splitkv(a["q"], a["k"], a["v"], a["mask"], a["total"], a["past"], a["out"],
                                a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["cap"], a["D"],
                                a["causal"], a["window"], a["scale"], a["softcap"], a["layout"],
                                a["planes"], a["dtype"], splits, lse, ws, ws_bytes, None)


def test_splitkv_validation(lib):
    assert call_splitkv(lib, -1) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 65) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 4, dtype=0) == attn.ATTN_ERR_UNSUPPORTED
    assert call_splitkv(lib, 4) == attn.ATTN_ERR_INVALID_ARG  # no workspace
    need = lib.attn_splitkv_workspace_bytes(2, 4, 200, 64, 4)
    assert need == 4 * 2 * 4 * 200 * 65 * 4
    assert call_splitkv(lib, 4, ws=0x78000000, ws_bytes=need - 4) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 4, ws=0x78000008, ws_bytes=need) == attn.ATTN_ERR_UNSUPPORTED
    assert call_splitkv(lib, 4, ws=Q, ws_bytes=need) == attn.ATTN_ERR_INVALID_ARG  # overlaps q
    assert call_splitkv(lib, 2, lse=0x7C000002) == attn.ATTN_ERR_UNSUPPORTED
    # the workspace and the log-sum-exp are written: they may overlap nothing the call reads
    WS, LSE = 0x78000000, 0x7C000000
    mask_kw = dict(mask=MASK, planes=2)
    assert call_splitkv(lib, 4, ws=MASK, ws_bytes=need, **mask_kw) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 4, ws=TOT - 16, ws_bytes=need, total=TOT) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 4, ws=PAST, ws_bytes=need, past=PAST) == attn.ATTN_ERR_INVALID_ARG
    assert call_splitkv(lib, 4, ws=WS, ws_bytes=need, lse=WS + need - 4) == attn.ATTN_ERR_INVALID_ARG
    for where in (Q, K + 4096, V, MASK + 64, TOT, PAST):
        assert call_splitkv(lib, 2, ws=WS, ws_bytes=need, lse=where, total=TOT, past=PAST,
                            **mask_kw) == attn.ATTN_ERR_INVALID_ARG, hex(where)
    assert lib.attn_splitkv_workspace_bytes(2, 4, 200, 64, 1) == 0
    assert call_splitkv(lib, 4, B=0) == attn.ATTN_OK
    assert call_splitkv(lib, 4, D=256) == attn.ATTN_ERR_UNSUPPORTED  # D 256: attn_fwd only
    assert call_splitkv(lib, 4, D=384) == attn.ATTN_ERR_UNSUPPORTED  # D 384: attn_fwd only


def test_valid_plane_counts_pass_validation_order(lib):
    # plane counts 1, B and B*Hq are accepted; with D=96 the request still
    # fails, but on the capability gate, proving the plane check passed
    for planes in (1, 2, 8):
        assert call(lib, mask=MASK, planes=planes, D=96) == attn.ATTN_ERR_UNSUPPORTED


def test_empty_problems_are_ok_without_touching_cuda(lib):
    assert call(lib, B=0, q=None, k=None, v=None, out=None) == attn.ATTN_OK
    assert call(lib, Sq=0) == attn.ATTN_OK


def test_selftest_rejects_bad_limits(lib):
    assert lib.attn_selftest_bounded_wait(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert lib.attn_selftest_bounded_wait(2_000_000_000, None) == attn.ATTN_ERR_INVALID_ARG


def test_set_wait_timeout(lib):
    assert lib.attn_set_wait_timeout_ns(5_000_000) == attn.ATTN_OK
    assert lib.attn_set_wait_timeout_ns(0) == attn.ATTN_OK  # back to the default


def test_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 2, 4, 64)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, torch.zeros(1, 1, 4, 32), torch.zeros(1, 1, 4, 32))
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q.double(), q.double())


def call_f32split(lib, ws=None, ws_bytes=0, **kw):
    a = dict(GOOD, **dict(dict(D=64), **kw))
    return lib.attn_fwd_f32_split(a["q"], a["k"], a["v"], a["mask"], a["total"], a["past"], a["out"],
                                  a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["cap"], a["D"],
                                  a["causal"], a["window"], a["scale"], a["softcap"], a["layout"],
                                  a["planes"], ws, ws_bytes, None)


def test_f32_split_validation(lib):
    need = lib.attn_f32_split_workspace_bytes(2, 2, 200, 64)
    assert need == 5 * 2 * 2 * 200 * 64 * 2  # k0, k1, k2, v0, v1 in bf16
    assert lib.attn_f32_split_workspace_bytes(0, 2, 200, 64) == 0
    WS = 0x7A000000
    assert call_f32split(lib) == attn.ATTN_ERR_INVALID_ARG                            # no workspace
    assert call_f32split(lib, ws=WS, ws_bytes=need - 1) == attn.ATTN_ERR_INVALID_ARG  # too small
    assert call_f32split(lib, ws=WS + 8, ws_bytes=need) == attn.ATTN_ERR_UNSUPPORTED  # misaligned
    assert call_f32split(lib, ws=K, ws_bytes=need) == attn.ATTN_ERR_INVALID_ARG       # overlaps k
    assert call_f32split(lib, ws=TOT, ws_bytes=need, total=TOT) == attn.ATTN_ERR_INVALID_ARG
    assert call_f32split(lib, ws=WS, ws_bytes=need, D=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call_f32split(lib, ws=WS, ws_bytes=need, D=256) == attn.ATTN_ERR_UNSUPPORTED
    assert call_f32split(lib, ws=WS, ws_bytes=need, Hq=5) == attn.ATTN_ERR_INVALID_ARG
    assert call_f32split(lib, ws=WS, ws_bytes=need, q=Q + 8) == attn.ATTN_ERR_UNSUPPORTED
    assert call_f32split(lib, ws=WS, ws_bytes=need, B=0) == attn.ATTN_OK              # empty problem
    # B * Hkv beyond the TMA plane coordinates of the four pieces
    assert call_f32split(lib, ws=WS, ws_bytes=2**62, B=40000, Hq=40000, Hkv=40000, Sq=1, Sk=1,
                         cap=1) == attn.ATTN_ERR_INVALID_ARG


# ---------------------------------------------------------------- dsa_index_select
DQ, DK, DW, DB, DO, DWS = (0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000)
DSA_GOOD = dict(query=DQ, key=DK, weights=DW, bias=DB, out=DO, B=2, S=8, H=16, D=64, T=300, top_k=32,
                scale=0.125, weights_scale=1.0, dtype=2, ws=DWS, ws_bytes=2 * 8 * 300 * 4 + 256)


def call_dsa(lib, **kw):
    a = dict(DSA_GOOD, **kw)
    return lib.dsa_index_select(a["query"], a["key"], a["weights"], a["bias"], a["out"], a["B"], a["S"],
                                a["H"], a["D"], a["T"], a["top_k"], a["scale"], a["weights_scale"],
                                a["dtype"], a["ws"], a["ws_bytes"], None)


def test_dsa_workspace_bytes(lib):
    assert lib.dsa_index_select_workspace_bytes(2, 8, 300) == 2 * 8 * 300 * 4 + 256  # scores, counter
    assert lib.dsa_index_select_workspace_bytes(0, 8, 300) == 0
    assert lib.dsa_index_select_workspace_bytes(2, 8, 0) == 0
    assert lib.dsa_index_select_workspace_bytes(-1, 8, 300) == 0


@pytest.mark.parametrize("case", [
    dict(dtype=3), dict(dtype=-1), dict(B=-1), dict(S=-1), dict(T=-1), dict(H=0), dict(D=0), dict(top_k=0),
    dict(scale=0.0), dict(scale=-1.0), dict(scale=math.inf), dict(scale=math.nan),
    dict(weights_scale=0.0), dict(weights_scale=math.nan),
    dict(query=None), dict(key=None), dict(weights=None), dict(bias=None), dict(out=None),
    dict(T=0, key=None, bias=None, query=None),
    dict(ws=None), dict(ws_bytes=2 * 8 * 300 * 4 + 255),
    dict(out=DQ + 64), dict(out=DB), dict(ws=DK), dict(ws=DO - 16),
    dict(B=2**20, S=2**20, T=2**20),
])
def test_dsa_invalid_arguments(lib, case):
    assert call_dsa(lib, **case) == attn.ATTN_ERR_INVALID_ARG, case


@pytest.mark.parametrize("case", [
    dict(H=65), dict(query=DQ + 1), dict(key=DK + 2, dtype=0), dict(bias=DB + 2), dict(out=DO + 4),
    dict(ws=DWS + 8),
])
def test_dsa_unsupported(lib, case):
    assert call_dsa(lib, **case) == attn.ATTN_ERR_UNSUPPORTED, case


def test_dsa_empty_problems_are_ok(lib):
    assert call_dsa(lib, B=0) == attn.ATTN_OK
    assert call_dsa(lib, S=0, query=None, out=None) == attn.ATTN_OK
    assert call_dsa(lib, T=0, key=None, bias=None, ws=None, ws_bytes=0, H=65) == attn.ATTN_ERR_UNSUPPORTED


def test_dsa_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 2, 3, 8, dtype=torch.bfloat16)
    k = torch.zeros(1, 5, 8, dtype=torch.bfloat16)
    w = torch.zeros(1, 2, 3, dtype=torch.bfloat16)
    b = torch.zeros(1, 1, 2, 5)
    with pytest.raises(ValueError):
        attn.dsa_index_select(q, k.float(), w, b, top_k=2, scale=1.0)       # mixed dtypes
    with pytest.raises(ValueError):
        attn.dsa_index_select(q, k, w, b.half(), top_k=2, scale=1.0)        # bias not f32
    with pytest.raises(ValueError):
        attn.dsa_index_select(q, k[:, :4], w, b, top_k=2, scale=1.0)        # T mismatch
    with pytest.raises(ValueError):
        attn.dsa_index_select(q[0], k, w, b, top_k=2, scale=1.0)            # rank


# attn_fwd_host: host buffers (fake addresses: never read before validation
# passes) plus device buffers of the same sizes
HQ, HK, HV, HOUT, HMASK, HTOT, HPAST = (0x11000000, 0x21000000, 0x31000000, 0x41000000, 0x51000000,
                                        0x61000000, 0x71000000)


def call_host(lib, hmask=None, htot=None, hpast=None, **kw):
    a = dict(GOOD, **kw)
    copied = (ctypes.c_uint64 * 2)(7, 7)
    rc = lib.attn_fwd_host(HQ, HK, HV, hmask, htot, hpast, HOUT,
                           a["q"], a["k"], a["v"], a["mask"], a["total"], a["past"], a["out"],
                           a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["cap"], a["D"], a["causal"],
                           a["window"], a["scale"], a["softcap"], a["layout"], a["planes"], a["dtype"],
                           None, copied)
    return rc, (copied[0], copied[1])


@pytest.mark.parametrize("case", ["dtype", "Hq_not_multiple", "Sk_over_capacity", "nan_scale",
                                  "bad_plane_count", "out_overlaps_q", "null_out"])
def test_host_entry_validates_like_attn_fwd(lib, case):
    """attn_fwd_host checks the whole problem as attn_fwd would, on its device
    buffers, before any copy or CUDA call; nothing is reported copied."""
    kw = dict(INVALID[case])
    hm = HMASK if kw.get("mask") else None
    rc, copied = call_host(lib, hmask=hm, **kw)
    assert rc == attn.ATTN_ERR_INVALID_ARG
    assert copied == (0, 0)


def test_host_entry_pairs_host_and_device_buffers(lib):
    """A mask or length array must be given on both sides or on neither."""
    assert call_host(lib, hmask=HMASK)[0] == attn.ATTN_ERR_INVALID_ARG          # no device mask
    assert call_host(lib, mask=MASK, planes=2)[0] == attn.ATTN_ERR_INVALID_ARG  # no host mask
    assert call_host(lib, htot=HTOT)[0] == attn.ATTN_ERR_INVALID_ARG
    assert call_host(lib, past=PAST)[0] == attn.ATTN_ERR_INVALID_ARG


def test_host_entry_unsupported_and_empty(lib):
    assert call_host(lib, D=96)[0] == attn.ATTN_ERR_UNSUPPORTED
    assert call_host(lib, B=0, q=None, k=None, v=None, out=None) == (attn.ATTN_OK, (0, 0))
