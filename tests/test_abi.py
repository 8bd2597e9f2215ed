"""The C ABI without a GPU: the library loads, exports every function
include/rf.h declares, and rejects invalid arguments on the host (no CUDA
call is made before validation, so these run on a machine without a GPU)."""

import ctypes
import math
import os
import re

import pytest

from online_softmax_attention_rf_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rf.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return api.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for required in ("rf_softmax_rows", "rf_attn_fwd", "rf_attn_decode_splitk",
                     "rf_splitk_merge"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    names = _declared()
    assert names
    for n in names:
        assert hasattr(L, n), n
    # the binding mirrors the header one to one
    assert sorted(api.SIGNATURES) == names


def test_version_and_workspace_size(L):
    assert L.rf_version() == 1
    n = 16 * 32 * 32 * 129 * 4
    assert api.decode_workspace_bytes(16, 32, 32, 128) == (n + 255) // 256 * 256
    assert api.decode_workspace_bytes(0, 32, 32, 128) == 0


A = 0x10000        # a 16-byte-aligned fake device address; never dereferenced
MIS = 0x10008      # misaligned for TMA


def _attn(L, q=A, k=A, v=A, o=A, lse=A, B=1, H=4, Hkv=2, Sq=256, Sk=256, d=128, scale=0.1,
          causal=0, bm=None, dt=api.RF_BF16):
    return L.rf_attn_fwd(q, k, v, o, lse, B, H, Hkv, Sq, Sk, d, scale, causal, bm, dt, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(Hkv=3), api.RF_ERR_INVALID),               # H % Hkv
    (dict(scale=0.0), api.RF_ERR_INVALID),
    (dict(scale=-1.0), api.RF_ERR_INVALID),
    (dict(scale=math.nan), api.RF_ERR_INVALID),
    (dict(scale=math.inf), api.RF_ERR_INVALID),
    (dict(causal=2), api.RF_ERR_INVALID),
    (dict(B=0), api.RF_ERR_INVALID),
    (dict(Sq=-1), api.RF_ERR_INVALID),
    (dict(Sq=(1 << 30) + 1), api.RF_ERR_INVALID),       # row indices stay 32-bit
    (dict(Sk=(1 << 30) + 1), api.RF_ERR_INVALID),
    (dict(d=96), api.RF_ERR_UNSUPPORTED),            # bf16 head dims: 64, 128
    (dict(d=258, dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
    (dict(d=66, dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
    (dict(dt=7), api.RF_ERR_INVALID),
    (dict(q=None), api.RF_ERR_INVALID),
    (dict(k=None), api.RF_ERR_INVALID),
    (dict(o=None), api.RF_ERR_INVALID),
    (dict(q=MIS), api.RF_ERR_INVALID),
    (dict(v=MIS), api.RF_ERR_INVALID),
    (dict(lse=A + 2), api.RF_ERR_INVALID),
])
def test_attn_fwd_rejects(L, kw, expect):
    assert _attn(L, **kw) == expect
    assert L.rf_last_error()


def _rowwise(L, q=A, k=A, v=A, o=A, lse=A, B=1, H=4, Hkv=2, Sq=256, Sk=256, d=128, scale=0.1,
             causal=0, bm=None, dt=api.RF_BF16):
    return L.rf_attn_fwd_rowwise(q, k, v, o, lse, B, H, Hkv, Sq, Sk, d, scale, causal, bm, dt, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(Hkv=3), api.RF_ERR_INVALID),
    (dict(scale=0.0), api.RF_ERR_INVALID),
    (dict(scale=math.nan), api.RF_ERR_INVALID),
    (dict(causal=2), api.RF_ERR_INVALID),
    (dict(B=0), api.RF_ERR_INVALID),
    (dict(Sk=(1 << 30) + 1), api.RF_ERR_INVALID),
    (dict(d=32, dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),   # row-wise head dims: 64, 128
    (dict(d=256, dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
    (dict(d=96), api.RF_ERR_UNSUPPORTED),
    (dict(dt=7), api.RF_ERR_INVALID),
    (dict(q=None), api.RF_ERR_INVALID),
    (dict(v=MIS), api.RF_ERR_INVALID),
    (dict(lse=A + 2), api.RF_ERR_INVALID),
])
def test_attn_fwd_rowwise_rejects(L, kw, expect):
    # the row-wise entry shares rf_attn_fwd's checks, all before any CUDA call
    assert _rowwise(L, **kw) == expect
    assert L.rf_last_error()


def test_attn_fwd_rowwise_rejects_bad_blockmask(L):
    bm = api.RFBlockMask(128, 128, 2, 2, A, A, 0)
    bm.nqt = 3
    assert _rowwise(L, bm=ctypes.byref(bm)) == api.RF_ERR_INVALID
    assert _rowwise(L, q=None, o=None, Sq=0) == api.RF_OK   # no query rows: nothing to do


def test_decode_workspace_size_formula(L):
    # o_part [B*H, nsplit, d] then lse_part [B*H, nsplit], float32, rounded up to 256 bytes
    for B, H, nsplit, d in [(1, 1, 1, 64), (3, 5, 7, 128), (16, 32, 32, 128), (2, 128, 16, 512)]:
        n = B * H * nsplit * (d + 1) * 4
        assert L.rf_decode_workspace_bytes(B, H, nsplit, d) == (n + 255) // 256 * 256
    for bad in [(0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 0)]:
        assert L.rf_decode_workspace_bytes(*bad) == 0
    assert L.rf_mla_decode_workspace_bytes(2, 16) == L.rf_decode_workspace_bytes(2, 128, 16, 512)


def test_attn_fwd_empty_query_is_a_no_op(L):
    assert _attn(L, q=None, o=None, Sq=0) == api.RF_OK


@pytest.mark.parametrize("field,value", [
    ("tile_q", 64), ("tile_k", 256), ("nqt", 3), ("nkt", 1), ("per_head", 2), ("row_ptr", 0),
    ("col_idx", 0)])
def test_attn_fwd_rejects_bad_blockmask(L, field, value):
    bm = api.RFBlockMask(128, 128, 2, 2, A, A, 0)
    setattr(bm, field, value)
    assert _attn(L, bm=ctypes.byref(bm)) == api.RF_ERR_INVALID


def _decode(L, q=A, k=A, v=A, o=A, lse=A, B=2, H=8, Hkv=2, Sk=1000, d=128, scale=0.1, nsplit=4,
            ws=A, ws_bytes=None, dt=api.RF_BF16):
    if ws_bytes is None:
        ws_bytes = api.decode_workspace_bytes(B, H, nsplit, d)
    return L.rf_attn_decode_splitk(q, k, v, o, lse, B, H, Hkv, Sk, d, scale, nsplit, ws, ws_bytes,
                                   dt, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(nsplit=0), api.RF_ERR_INVALID),
    (dict(nsplit=1001), api.RF_ERR_INVALID),        # more splits than keys
    (dict(ws_bytes=16), api.RF_ERR_INVALID),
    (dict(ws=None), api.RF_ERR_INVALID),
    (dict(ws=MIS), api.RF_ERR_INVALID),
    (dict(Hkv=3), api.RF_ERR_INVALID),
    (dict(H=64, Hkv=2), api.RF_ERR_UNSUPPORTED),    # 32 query heads per kv head
    (dict(dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
    (dict(d=96), api.RF_ERR_UNSUPPORTED),
    (dict(scale=0.0), api.RF_ERR_INVALID),
    (dict(Sk=0), api.RF_ERR_INVALID),
])
def test_decode_rejects(L, kw, expect):
    assert _decode(L, **kw) == expect


def _decode_noalloc(L, q=A, k=A, v=A, o=A, lse=A, B=2, H=8, Hkv=2, Sk=1000, d=128, scale=0.1,
                    nsplit=4, dt=api.RF_BF16):
    return L.rf_attn_decode_splitk_noalloc(q, k, v, o, lse, B, H, Hkv, Sk, d, scale, nsplit, dt,
                                           None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), api.RF_ERR_INVALID),
    (dict(k=None), api.RF_ERR_INVALID),
    (dict(v=None), api.RF_ERR_INVALID),
    (dict(o=None), api.RF_ERR_INVALID),
    (dict(q=MIS), api.RF_ERR_INVALID),
    (dict(lse=A + 2), api.RF_ERR_INVALID),
    (dict(Hkv=3), api.RF_ERR_INVALID),               # H % Hkv
    (dict(nsplit=0), api.RF_ERR_INVALID),
    (dict(nsplit=1001), api.RF_ERR_INVALID),         # more splits than keys
    (dict(B=0), api.RF_ERR_INVALID),                 # would need no workspace at all
    (dict(scale=math.nan), api.RF_ERR_INVALID),
    (dict(dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
    (dict(d=96), api.RF_ERR_UNSUPPORTED),
    (dict(H=64, Hkv=2), api.RF_ERR_UNSUPPORTED),
    # partials of 64 x 32 rows x 64 splits x 129 floats: 67.6 MB > the 16 MiB array
    (dict(B=64, H=32, Hkv=8, Sk=65536, nsplit=64), api.RF_ERR_INVALID),
])
def test_decode_noalloc_rejects_before_any_cuda_call(L, kw, expect):
    # on a machine without a GPU any CUDA call would give RF_ERR_CUDA instead
    assert _decode_noalloc(L, **kw) == expect
    assert L.rf_last_error().decode().startswith("rf_attn_decode_splitk_noalloc")


@pytest.mark.parametrize("args,expect", [
    ((A, A, A, A, 5, 0, 64, api.RF_BF16), api.RF_ERR_INVALID),      # nsplit 0
    ((A, A, A, A, 5, 4, 2048, api.RF_BF16), api.RF_ERR_INVALID),    # d > 1024
    ((A, A, A, A, -1, 4, 64, api.RF_BF16), api.RF_ERR_INVALID),
    ((None, A, A, A, 5, 4, 64, api.RF_BF16), api.RF_ERR_INVALID),
    ((A, A, A, A, 0, 4, 64, api.RF_BF16), api.RF_OK),               # no rows: no launch
])
def test_merge_validation(L, args, expect):
    o_part, lse_part, o, lse, rows, nsplit, d, dt = args
    assert L.rf_splitk_merge(o_part, lse_part, o, lse, rows, nsplit, d, dt, None) == expect


def test_softmax_and_blockmask_validation(L):
    assert L.rf_softmax_rows(A, A, -1, 5, api.RF_F32, None) == api.RF_ERR_INVALID
    assert L.rf_softmax_rows(A, A, 5, 5, 9, None) == api.RF_ERR_INVALID
    assert L.rf_softmax_rows(None, A, 5, 5, api.RF_F32, None) == api.RF_ERR_INVALID
    assert L.rf_softmax_rows(A, A, 0, 5, api.RF_F32, None) == api.RF_OK
    assert L.rf_blockmask_build(A, 1, 4, 0, A, A, 16, None) == api.RF_ERR_INVALID
    assert L.rf_blockmask_build(None, 1, 4, 4, A, A, 16, None) == api.RF_ERR_INVALID
    assert L.rf_blockmask_build(A, 1, 4, 4, A, A, -1, None) == api.RF_ERR_INVALID
    assert L.rf_debug_set_visited(A, 0) == api.RF_ERR_INVALID
    assert L.rf_debug_set_visited(None, 0) == api.RF_OK
    assert L.rf_device_status(None, None) == api.RF_ERR_INVALID


def _attn_host(L, q=A, k=A, v=A, o=A, lse=A, B=2, H=4, Hkv=2, Sq=256, Sk=256, d=128, ws=0x20000,
               ws_bytes=None, dt=api.RF_BF16):
    if ws_bytes is None:
        ws_bytes = L.rf_attn_fwd_host_workspace_bytes(B, H, Hkv, Sq, Sk, d, dt)
    return L.rf_attn_fwd_host(q, k, v, o, lse, B, H, Hkv, Sq, Sk, d, 0.1, 0, None, dt, ws,
                              ws_bytes, None)


def test_attn_fwd_host_workspace_size(L):
    # two chunks in flight, each 256-byte aligned Q, K, V, O and LSE of one
    # (batch, kv-head group) slice: B = 2 -> 4 chunks per batch element -> 1 kv head
    n = L.rf_attn_fwd_host_workspace_bytes(2, 4, 4, 256, 512, 128, api.RF_BF16)
    slot = 256 * 128 * 2 + 2 * 512 * 128 * 2 + 256 * 128 * 2 + 256 * 4
    assert n == 2 * slot
    assert L.rf_attn_fwd_host_workspace_bytes(0, 4, 4, 256, 512, 128, api.RF_BF16) == 0
    assert L.rf_attn_fwd_host_workspace_bytes(1, 4, 3, 256, 512, 128, api.RF_BF16) == 0
    assert L.rf_attn_fwd_host_workspace_bytes(1, 4, 4, 256, 512, 128, 7) == 0


@pytest.mark.parametrize("kw", [
    dict(B=0), dict(Hkv=3), dict(dt=9), dict(q=None), dict(k=None), dict(o=None),
    dict(ws=None), dict(ws=0x20008), dict(ws_bytes=1024)])
def test_attn_fwd_host_rejects(L, kw):
    assert _attn_host(L, **kw) == api.RF_ERR_INVALID


def test_two_level_validation(L):
    """Two-level masks: the builder and rf_attn_fwd reject bad arguments on
    the host (no device memory is touched)."""
    b = L.rf_blockmask_build_elements
    assert b(A, 0, 10, 10, A, A, A, A, 4, None, None) == api.RF_ERR_INVALID      # nheads
    assert b(A, 1, 0, 10, A, A, A, A, 4, None, None) == api.RF_ERR_INVALID      # Sq
    assert b(None, 1, 10, 10, A, A, A, A, 4, None, None) == api.RF_ERR_INVALID  # dense
    assert b(A, 1, 10, 10, A, A, None, A, 4, None, None) == api.RF_ERR_INVALID  # tile_bits
    assert b(A, 1, 10, 10, A, A, A, A + 4, 4, None, None) == api.RF_ERR_INVALID  # bits align
    assert b(A, 1, 10, 10, A, A, A, A, -1, None, None) == api.RF_ERR_INVALID    # bits_cap
    bm = api.RFBlockMask(128, 128, 2, 2, A, A, 0, A, None)                      # bits missing
    assert _attn(L, bm=ctypes.byref(bm)) == api.RF_ERR_INVALID


def test_fault_injection_sites(L):
    assert L.rf_debug_inject_fault(7) == api.RF_ERR_INVALID
    assert L.rf_debug_inject_fault(1) == api.RF_OK
    assert L.rf_debug_inject_fault(0) == api.RF_OK


@pytest.mark.parametrize("kw", [
    dict(T=-1), dict(E=0), dict(E=1025), dict(k=0), dict(k=33, E=64), dict(k=9, E=8),
    dict(renorm=2), dict(dt=9), dict(logits=None), dict(idx=None), dict(w=None)])
def test_moe_route_rejects(L, kw):
    a = dict(logits=A, T=16, E=64, k=8, renorm=0, idx=A, w=A, lse=None, dt=api.RF_BF16)
    a.update(kw)
    assert L.rf_moe_route(a["logits"], a["T"], a["E"], a["k"], a["renorm"], a["idx"], a["w"],
                          a["lse"], a["dt"], None) == api.RF_ERR_INVALID


def test_moe_route_and_moments_empty_are_no_ops(L):
    assert L.rf_moe_route(None, 0, 64, 8, 0, None, None, None, api.RF_F32, None) == api.RF_OK
    assert L.rf_row_moments(None, 0, 64, 1e-5, None, None, None, api.RF_F32, None) == api.RF_OK
    assert L.rf_row_moments(None, 4, 0, 1e-5, None, None, None, api.RF_F32, None) == api.RF_OK


@pytest.mark.parametrize("rows,cols,eps,x,dt", [
    (-1, 4, 1e-5, A, api.RF_F32), (4, -1, 1e-5, A, api.RF_F32), (4, 4, -1.0, A, api.RF_F32),
    (4, 4, float("nan"), A, api.RF_F32), (4, 4, float("inf"), A, api.RF_F32),
    (4, 4, 1e-5, None, api.RF_F32), (4, 4, 1e-5, A, 9), (2 ** 31, 4, 1e-5, A, api.RF_F32)])
def test_row_moments_rejects(L, rows, cols, eps, x, dt):
    assert L.rf_row_moments(x, rows, cols, eps, A, A, None, dt, None) == api.RF_ERR_INVALID


def test_moment_of_inertia_validation(L):
    f = L.rf_moment_of_inertia
    assert f(A, A, -1, 4, A, A, A, None) == api.RF_ERR_INVALID
    assert f(A, A, 4, -1, A, A, A, None) == api.RF_ERR_INVALID
    assert f(None, A, 4, 4, A, A, A, None) == api.RF_ERR_INVALID
    assert f(A + 2, A, 4, 4, A, A, A, None) == api.RF_ERR_INVALID
    assert f(A, None, 2 ** 31, 4, A, A, A, None) == api.RF_ERR_INVALID
    assert f(None, None, 0, 4, None, None, None, None) == api.RF_OK


def test_fp8_validation(L):
    q = L.rf_rowquant_e4m3
    assert q(A, 4, 100, A, A, api.RF_BF16, None) == api.RF_ERR_UNSUPPORTED       # K % 16
    assert q(A, 4, 65536, A, A, api.RF_BF16, None) == api.RF_ERR_UNSUPPORTED     # > 64 KB
    assert q(A, 4, 64, A, A, 9, None) == api.RF_ERR_INVALID
    assert q(None, 4, 64, A, A, api.RF_BF16, None) == api.RF_ERR_INVALID
    assert q(MIS, 4, 64, A, A, api.RF_BF16, None) == api.RF_ERR_INVALID
    assert q(None, 0, 64, None, None, api.RF_BF16, None) == api.RF_OK
    g = L.rf_fp8_gemm
    assert g(A, A, A, A, A, 100, 256, 128, None) == api.RF_ERR_UNSUPPORTED
    assert g(A, A, A, A, A, 128, 128, 128, None) == api.RF_ERR_UNSUPPORTED
    assert g(A, A, A, A, A, 128, 256, 100, None) == api.RF_ERR_UNSUPPORTED
    assert g(None, A, A, A, A, 128, 256, 128, None) == api.RF_ERR_INVALID
    assert g(MIS, A, A, A, A, 128, 256, 128, None) == api.RF_ERR_INVALID
    assert g(None, None, None, None, None, 0, 256, 128, None) == api.RF_OK


def test_mla_decode_validation(L):
    ws = L.rf_mla_decode_workspace_bytes(2, 4)
    assert ws == (2 * 128 * 4 * 513 * 4 + 255) // 256 * 256
    f = L.rf_mla_decode
    assert f(A, A, A, A, 0, 64, 0.1, 1, A, ws, None) == api.RF_ERR_INVALID       # B
    assert f(A, A, A, A, 2, 64, 0.1, 65, A, ws, None) == api.RF_ERR_INVALID      # nsplit > Sk
    assert f(A, A, A, A, 2, 64, -1.0, 4, A, ws, None) == api.RF_ERR_INVALID      # scale
    assert f(None, A, A, A, 2, 64, 0.1, 4, A, ws, None) == api.RF_ERR_INVALID
    assert f(MIS, A, A, A, 2, 64, 0.1, 4, A, ws, None) == api.RF_ERR_INVALID
    assert f(A, A, A, A, 2, 64, 0.1, 4, A, ws - 256, None) == api.RF_ERR_INVALID  # workspace


def test_no_cpu_fallback(L, monkeypatch):
    """The binding computes nothing itself. Without the library every call
    raises, and host tensors are refused rather than computed on the CPU."""
    import torch
    x = torch.randn(4, 8)
    with pytest.raises(ValueError):
        api.softmax_rows(x)
    q = torch.randn(1, 1, 4, 64).to(torch.bfloat16)
    with pytest.raises(ValueError):
        api.attn_fwd(q, q, q)
    monkeypatch.setattr(api, "_LIB", None)
    monkeypatch.setattr(api, "library_path", lambda: os.path.join(ROOT, "no_such_dir", "librf.so"))
    with pytest.raises(RuntimeError):
        api.lib()
    with pytest.raises(RuntimeError):
        api.decode_workspace_bytes(1, 1, 1, 64)


@pytest.mark.parametrize("kw,expect", [
    (dict(ws=None), api.RF_ERR_INVALID),
    (dict(ws=MIS), api.RF_ERR_INVALID),
    (dict(ws_bytes=16), api.RF_ERR_INVALID),
    (dict(q=None), api.RF_ERR_INVALID),
    (dict(Hkv=3), api.RF_ERR_INVALID),
    (dict(nsplit=1001), api.RF_ERR_INVALID),
    (dict(dt=api.RF_F32), api.RF_ERR_UNSUPPORTED),
])
def test_decode_partials_rejects(L, kw, expect):
    a = dict(q=A, k=A, v=A, ws=A, ws_bytes=None, B=2, H=8, Hkv=2, Sk=1000, d=128, scale=0.1,
             nsplit=4, dt=api.RF_BF16)
    a.update(kw)
    if a["ws_bytes"] is None:
        a["ws_bytes"] = api.decode_workspace_bytes(a["B"], a["H"], a["nsplit"], a["d"])
    assert L.rf_attn_decode_partials(a["q"], a["k"], a["v"], a["ws"], a["ws_bytes"], a["B"],
                                     a["H"], a["Hkv"], a["Sk"], a["d"], a["scale"], a["nsplit"],
                                     a["dt"], None) == expect


@pytest.mark.parametrize("args,expect", [
    ((A, A, A, A, 5, 0, 64, 64, 0, 1, 5), api.RF_ERR_INVALID),        # nsplit 0
    ((A, A, A, A, 5, 4, 64, -64, 256, 1, 4), api.RF_ERR_INVALID),     # negative stride
    ((A, A, A, A, 5, 4, 64, 64, 256, 1, -1), api.RF_ERR_INVALID),
    ((None, A, A, A, 5, 4, 64, 64, 256, 1, 4), api.RF_ERR_INVALID),
    ((A, A, A, A + 2, 5, 4, 64, 64, 256, 1, 4), api.RF_ERR_INVALID),  # misaligned lse
    ((A, A, A, A, 0, 4, 64, 64, 256, 1, 4), api.RF_OK),               # no rows: no launch
])
def test_merge_strided_validation(L, args, expect):
    o_part, lse_part, o, lse, rows, nsplit, d, os_, or_, ls_, lr_ = args
    assert L.rf_splitk_merge_strided(o_part, lse_part, o, lse, rows, nsplit, d, os_, or_, ls_,
                                     lr_, api.RF_F32, None) == expect


def test_blockmask_counts_validation(L):
    f = L.rf_blockmask_counts
    assert f(None, 0, 1, 128, 128, 0, A, None) == api.RF_ERR_INVALID          # B
    assert f(None, 1, 1, -1, 128, 0, A, None) == api.RF_ERR_INVALID          # Sq
    assert f(None, 1, 1, 128, 128, 2, A, None) == api.RF_ERR_INVALID          # causal
    assert f(None, 1, 1, 128, 128, 0, None, None) == api.RF_ERR_INVALID       # counts
    assert f(None, 1, 1, 128, 128, 0, A + 4, None) == api.RF_ERR_INVALID      # alignment
    bm = api.RFBlockMask(128, 128, 2, 2, A, A, 0)
    assert f(ctypes.byref(bm), 1, 1, 128, 128, 0, A, None) == api.RF_ERR_INVALID  # nqt != 1
    bm = api.RFBlockMask(128, 128, 1, 1, None, A, 0)
    assert f(ctypes.byref(bm), 1, 1, 128, 128, 0, A, None) == api.RF_ERR_INVALID  # NULL lists
    bm = api.RFBlockMask(64, 128, 1, 1, A, A, 0)
    assert f(ctypes.byref(bm), 1, 1, 128, 128, 0, A, None) == api.RF_ERR_INVALID  # tile side


def test_blockmask_cta_order_validation(L):
    # every invalid argument is refused before any CUDA call
    f, n = L.rf_blockmask_cta_order, L.rf_blockmask_cta_order_len
    # items = B * H * ceil(ceil(nqt / 2) / 2)
    assert n(1, 1, 128) == 1 and n(2, 3, 2048) == 2 * 3 * 4 and n(1, 1, 640) == 2
    assert n(0, 1, 128) == 0 and n(1, 1, 0) == 0
    bm = api.RFBlockMask(128, 128, 16, 16, A, A, 0)
    ok = dict(bm=ctypes.byref(bm), B=1, H=1, Sq=2048, order=A, cap=4)
    def call(**kw):
        a = dict(ok); a.update(kw)
        return f(a["bm"], a["B"], a["H"], a["Sq"], a["order"], a["cap"], None)
    assert call(B=0) == api.RF_ERR_INVALID
    assert call(Sq=0) == api.RF_ERR_INVALID
    assert call(bm=None) == api.RF_ERR_INVALID
    assert call(order=None) == api.RF_ERR_INVALID
    assert call(order=A + 2) == api.RF_ERR_INVALID                            # alignment
    assert call(cap=3) == api.RF_ERR_INVALID                                  # 4 items needed
    assert call(Sq=1000) == api.RF_ERR_INVALID                                # nqt 8 != 16
    bad = api.RFBlockMask(128, 128, 16, 16, None, A, 0)
    assert call(bm=ctypes.byref(bad)) == api.RF_ERR_INVALID                   # no row_ptr
    bad = api.RFBlockMask(128, 128, 16, 16, A, A, 2)
    assert call(bm=ctypes.byref(bad)) == api.RF_ERR_INVALID                   # per_head
    assert L.rf_last_error()


def test_attn_fwd_rejects_misaligned_cta_order(L):
    bm = api.RFBlockMask(128, 128, 2, 2, A, A, 0, None, None, A + 2)
    assert _attn(L, bm=ctypes.byref(bm)) == api.RF_ERR_INVALID
