"""rf_attn_decode_splitk_noalloc: split-K decode with the library's own
static device workspace.

Some callers of this library cannot call cudaMalloc -- a plug-in running inside
a host process whose runtime owns all device memory, or a serving loop that
forbids allocation once it has started -- so they cannot hand
rf_attn_decode_splitk the workspace it needs for the per-split partials. The
allocation-free entry point takes that workspace from a fixed 16 MiB array in
the library's device image instead. This test calls it through the C ABI and
checks it against the allocating entry point, twice in a row (the array keeps
the previous call's partials, so the second call also shows that stale
contents do not leak into a new result), and checks that shapes needing more
than the array holds are refused.

The file name sorts last so that a run that stops at the first failure has
already run every other test.
"""

import ctypes
import math

import pytest
import torch

from online_softmax_attention_rf_gb300 import api, build, inputs
from tests.helpers import TOL_BF16_LSE, TOL_BF16_O, assert_close, f64

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


def _noalloc(L, q, k, v, nsplit):
    B, H, _, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, 1, dtype=torch.float32, device=q.device)
    st = L.rf_attn_decode_splitk_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), B, H, Hkv, Sk, d, 1.0 / math.sqrt(d), nsplit,
        api.RF_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == api.RF_OK, L.rf_last_error()
    return o, lse


def test_noalloc_decode_matches_the_allocating_entry_point(cuda_device):
    build.build()
    L = api.lib()
    # two calls in a row; the second is smaller, so stale partials of the first
    # remain in the shared array around the ones it writes
    for (B, H, Hkv, Sk, d, nsplit, seed) in [(16, 32, 8, 65536, 128, 32, 3),
                                            (2, 8, 2, 5000, 64, 7, 41)]:
        q, k, v = (t.cuda() for t in inputs.make_qkv(B, H, Hkv, 1, Sk, d, seed, "bf16"))
        assert api.decode_workspace_bytes(B, H, nsplit, d) <= STATIC_BYTES
        o_ref, lse_ref = api.attn_decode_splitk(q, k, v, nsplit)
        o, lse = _noalloc(L, q, k, v, nsplit)
        torch.cuda.synchronize()
        assert api.device_status() == 0
        assert_close(o, f64(o_ref), TOL_BF16_O, "O")
        assert_close(lse, f64(lse_ref), TOL_BF16_LSE, "LSE")


def test_noalloc_decode_refuses_shapes_beyond_the_static_workspace(cuda_device):
    L = api.lib()
    # B=64, H=64, nsplit=64, d=128: 4 * 64*64*64*129 bytes = 135 MB > 16 MiB
    q = torch.zeros(64, 64, 1, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(64, 8, 64, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    st = L.rf_attn_decode_splitk_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(o.data_ptr()), None, 64, 64, 8, 64, 128,
        0.1, 64, api.RF_BF16, None)
    assert st == api.RF_ERR_INVALID
    assert b"static workspace" in L.rf_last_error()
