"""Thin ctypes binding of librf.so (declared in include/rf.h).

Argument marshalling only: each function checks that its torch tensors are
CUDA, contiguous and of the right dtype, passes their data pointers, sizes
and the current CUDA stream to the C entry point of the same name, and turns
a non-OK status into ``RFError``. Every step of the computation runs in the
library's kernels; nothing here computes, and there is no CPU fallback -- if
the library is missing, every call raises.
"""

import ctypes
import math
import os

import torch

from . import build as _build

RF_OK, RF_ERR_INVALID, RF_ERR_UNSUPPORTED, RF_ERR_CUDA, RF_ERR_TIMEOUT = range(5)
RF_F32, RF_BF16 = 0, 1
RF_KERNEL_BLOCKWISE, RF_KERNEL_ROWWISE = 0, 1
_STATUS_NAMES = {0: "RF_OK", 1: "RF_ERR_INVALID", 2: "RF_ERR_UNSUPPORTED", 3: "RF_ERR_CUDA",
                 4: "RF_ERR_TIMEOUT"}
TILE = 128


class RFError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (_STATUS_NAMES.get(status, status), message))
        self.status = status


class RFBlockMask(ctypes.Structure):
    _fields_ = [("tile_q", ctypes.c_int), ("tile_k", ctypes.c_int), ("nqt", ctypes.c_int),
                ("nkt", ctypes.c_int), ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p),
                ("per_head", ctypes.c_int), ("tile_bits", ctypes.c_void_p),
                ("bits", ctypes.c_void_p), ("cta_order", ctypes.c_void_p)]


_LIB = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name: (restype, argtypes) -- mirrors include/rf.h
SIGNATURES = {
    "rf_softmax_rows": (_I, [_P, _P, _I64, _I64, _I, _P]),
    "rf_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                         ctypes.POINTER(RFBlockMask), _I, _P]),
    "rf_attn_decode_splitk": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _I,
                                   _P]),
    "rf_attn_decode_splitk_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I,
                                           _P]),
    "rf_attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                              ctypes.POINTER(RFBlockMask), _I, _P, _SZ, _P]),
    "rf_attn_fwd_host_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "rf_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "rf_splitk_merge": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _P]),
    "rf_attn_decode_partials": (_I, [_P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I, _I, _I, _F,
                                     _I, _I, _P]),
    "rf_splitk_merge_strided": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I64, _I64, _I64, _I64, _I,
                                     _P]),
    "rf_blockmask_build": (_I, [_P, _I, _I, _I, _P, _P, _I64, _P]),
    "rf_blockmask_build_elements": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _I64, _P, _P]),
    "rf_blockmask_counts": (_I, [ctypes.POINTER(RFBlockMask), _I, _I, _I, _I, _I, _P, _P]),
    "rf_blockmask_cta_order_len": (_I64, [_I, _I, _I]),
    "rf_blockmask_cta_order": (_I, [ctypes.POINTER(RFBlockMask), _I, _I, _I, _P, _I64, _P]),
    "rf_attn_fwd_rowwise": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I,
                                 ctypes.POINTER(RFBlockMask), _I, _P]),
    "rf_attn_choose_kernel": (_I, [_I, _I, _I, _I, _I, _I64, _I64, _I64, _I]),
    "rf_attn_estimate_us": (_I, [_I, _I, _I, _I, _I, _I64, _I64, _I64, _I,
                                 ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
    "rf_moe_route": (_I, [_P, _I64, _I, _I, _I, _P, _P, _P, _I, _P]),
    "rf_row_moments": (_I, [_P, _I64, _I64, _F, _P, _P, _P, _I, _P]),
    "rf_moment_of_inertia": (_I, [_P, _P, _I64, _I64, _P, _P, _P, _P]),
    "rf_rowquant_e4m3": (_I, [_P, _I64, _I64, _P, _P, _I, _P]),
    "rf_mla_decode_workspace_bytes": (_SZ, [_I, _I]),
    "rf_mla_decode": (_I, [_P, _P, _P, _P, _I, _I, _F, _I, _P, _SZ, _P]),
    "rf_fp8_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "rf_debug_set_visited": (_I, [_P, _I64]),
    "rf_debug_inject_fault": (_I, [_I]),
    "rf_device_status": (_I, [_P, ctypes.POINTER(_I)]),
    "rf_last_error": (ctypes.c_char_p, []),
    "rf_version": (_I, []),
}


def library_path():
    return _build.LIB_PATH


def lib():
    """The loaded librf.so; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                "librf.so is not built (%s); run `python -m online_softmax_attention_rf_gb300.build`"
                % path)
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _check(status):
    if status != RF_OK:
        raise RFError(status, lib().rf_last_error().decode(errors="replace"))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dt(t):
    if t.dtype == torch.float32:
        return RF_F32
    if t.dtype == torch.bfloat16:
        return RF_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


class BlockMask:
    """Block-sparse 128 x 128 tile lists resident on the device.

    ``row_ptr`` int32 [nheads*nqt + 1] and ``col_idx`` int32 [capacity];
    ``per_head`` is 1 when each (batch, head) has its own lists. With the
    two-level form, ``tile_bits`` int32 (parallel to ``col_idx``, -1 = full
    tile) and ``bits`` uint64 viewed as int64 [partial tiles, 256].
    ``cta_orders`` caches the tensor-core kernel's work order
    (rf_blockmask_cta_order) per (B, H, Sq).
    """

    def __init__(self, row_ptr, col_idx, nqt, nkt, per_head, tile_bits=None, bits=None):
        self.row_ptr, self.col_idx = row_ptr, col_idx
        self.nqt, self.nkt, self.per_head = nqt, nkt, per_head
        self.tile_bits, self.bits = tile_bits, bits
        self.cta_orders = {}

    def as_struct(self, order=None):
        return RFBlockMask(TILE, TILE, self.nqt, self.nkt, self.row_ptr.data_ptr(),
                           self.col_idx.data_ptr(), self.per_head,
                           self.tile_bits.data_ptr() if self.tile_bits is not None else None,
                           self.bits.data_ptr() if self.bits is not None else None,
                           order.data_ptr() if order is not None else None)

    def cta_order(self, B, H, Sq):
        """rf_blockmask_cta_order for an attention of B x H heads and Sq queries:
        computed on the current stream the first time, then cached (the
        kernel reads one entry per CTA)."""
        key = (B, H, Sq)
        if key not in self.cta_orders:
            n = int(lib().rf_blockmask_cta_order_len(B, H, Sq))
            order = torch.empty(max(1, n), dtype=torch.int32, device=self.row_ptr.device)
            bm = self.as_struct()
            _check(lib().rf_blockmask_cta_order(ctypes.byref(bm), B, H, Sq, _ptr(order), n,
                                                _stream()))
            self.cta_orders[key] = order
        return self.cta_orders[key]

    @classmethod
    def from_dense_elements(cls, elem_mask, device="cuda"):
        """Two-level lists (outer tiles + inner 8x8 bitmaps) from a bool/uint8
        element mask [Sq, Sk] (shared) or [nheads, Sq, Sk] (per head), built
        on the device (rf_blockmask_build_elements; a first pass counts the
        partial tiles to size the bitmaps)."""
        em = torch.as_tensor(elem_mask)
        per_head = 1 if em.dim() == 3 else 0
        if em.dim() == 2:
            em = em.unsqueeze(0)
        nheads, Sq, Sk = em.shape
        dense = em.to(device=device, dtype=torch.uint8).contiguous()
        nqt, nkt = -(-Sq // TILE), -(-Sk // TILE)
        row_ptr = torch.empty(nheads * nqt + 1, dtype=torch.int32, device=device)
        col_idx = torch.empty(nheads * nqt * nkt, dtype=torch.int32, device=device)
        tile_bits = torch.empty(nheads * nqt * nkt, dtype=torch.int32, device=device)
        n_partial = torch.zeros(1, dtype=torch.int32, device=device)
        blockmask_build_elements(dense, row_ptr, col_idx, tile_bits, None, n_partial)
        bits = torch.empty((max(1, int(n_partial.item())), 256), dtype=torch.int64, device=device)
        blockmask_build_elements(dense, row_ptr, col_idx, tile_bits, bits, n_partial)
        return cls(row_ptr, col_idx, nqt, nkt, per_head, tile_bits, bits)

    @classmethod
    def from_dense(cls, tile_mask, device="cuda"):
        """Build the lists on the device from a bool/uint8 mask [nqt, nkt] or
        [nheads, nqt, nkt] (rf_blockmask_build)."""
        tm = torch.as_tensor(tile_mask)
        per_head = 1 if tm.dim() == 3 else 0
        if tm.dim() == 2:
            tm = tm.unsqueeze(0)
        nheads, nqt, nkt = tm.shape
        dense = tm.to(device=device, dtype=torch.uint8).contiguous()
        row_ptr = torch.empty(nheads * nqt + 1, dtype=torch.int32, device=device)
        col_idx = torch.empty(max(1, nheads * nqt * nkt), dtype=torch.int32, device=device)
        blockmask_build(dense, row_ptr, col_idx)
        return cls(row_ptr, col_idx, nqt, nkt, per_head)


def blockmask_build(dense_u8, row_ptr, col_idx):
    """rf_blockmask_build on [nheads, nqt, nkt] uint8 -> row_ptr, col_idx (in place)."""
    _cuda(dense_u8, row_ptr, col_idx)
    nheads, nqt, nkt = dense_u8.shape
    _check(lib().rf_blockmask_build(_ptr(dense_u8), nheads, nqt, nkt, _ptr(row_ptr),
                                    _ptr(col_idx), col_idx.numel(), _stream()))


def blockmask_build_elements(dense_u8, row_ptr, col_idx, tile_bits, bits, n_partial=None):
    """rf_blockmask_build_elements on [nheads, Sq, Sk] uint8 (in place); ``bits``
    None builds the lists only (and counts the partial tiles into n_partial)."""
    _cuda(dense_u8, row_ptr, col_idx, tile_bits, bits, n_partial)
    nheads, Sq, Sk = dense_u8.shape
    cap = 0 if bits is None else bits.shape[0]
    _check(lib().rf_blockmask_build_elements(_ptr(dense_u8), nheads, Sq, Sk, _ptr(row_ptr),
                                             _ptr(col_idx), _ptr(tile_bits), _ptr(bits), cap,
                                             _ptr(n_partial), _stream()))


def softmax_rows(x, out=None):
    """rf_softmax_rows: softmax over the last dim of a 2-D float32/bf16 tensor."""
    _cuda(x)
    if x.dim() != 2:
        raise ValueError("x must be [rows, cols]")
    y = torch.empty_like(x) if out is None else out
    _cuda(y)
    _check(lib().rf_softmax_rows(_ptr(x), _ptr(y), x.shape[0], x.shape[1], _dt(x), _stream()))
    return y


def moe_route(logits, k, renorm=False, with_lse=True):
    """rf_moe_route: logits [T, E] -> (idx int32 [T, k], w float32 [T, k], lse or None)."""
    _cuda(logits)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    lse = torch.empty(T, dtype=torch.float32, device=logits.device) if with_lse else None
    _check(lib().rf_moe_route(_ptr(logits), T, E, int(k), 1 if renorm else 0, _ptr(idx), _ptr(w),
                              _ptr(lse), _dt(logits), _stream()))
    return idx, w, lse


def row_moments(x, eps=1e-5, normalize=True, out=None):
    """rf_row_moments: x [rows, cols] -> (mean, var, y or None), mean/var float32."""
    _cuda(x)
    if x.dim() != 2:
        raise ValueError("x must be [rows, cols]")
    rows = x.shape[0]
    mean = torch.empty(rows, dtype=torch.float32, device=x.device)
    var = torch.empty(rows, dtype=torch.float32, device=x.device)
    y = None
    if normalize:
        y = torch.empty_like(x) if out is None else out
        _cuda(y)
        if y.shape != x.shape or y.dtype != x.dtype:
            raise ValueError("out must match x")
    _check(lib().rf_row_moments(_ptr(x), rows, x.shape[1], float(eps), _ptr(mean), _ptr(var),
                                _ptr(y), _dt(x), _stream()))
    return mean, var, y


def moment_of_inertia(points, masses=None):
    """rf_moment_of_inertia: points [sets, n, 3] float32 (+ masses [sets, n])
    -> (total mass [sets], centre [sets, 3], inertia [sets])."""
    _cuda(points, masses)
    if points.dim() != 3 or points.shape[2] != 3 or points.dtype != torch.float32:
        raise ValueError("points must be float32 [sets, n, 3]")
    sets, n = points.shape[0], points.shape[1]
    if masses is not None and (masses.shape != (sets, n) or masses.dtype != torch.float32):
        raise ValueError("masses must be float32 [sets, n]")
    total = torch.empty(sets, dtype=torch.float32, device=points.device)
    centre = torch.empty(sets, 3, dtype=torch.float32, device=points.device)
    inertia = torch.empty(sets, dtype=torch.float32, device=points.device)
    _check(lib().rf_moment_of_inertia(_ptr(points), _ptr(masses), sets, n, _ptr(total),
                                      _ptr(centre), _ptr(inertia), _stream()))
    return total, centre, inertia


def rowquant_e4m3(x):
    """rf_rowquant_e4m3: x [rows, K] float32/bf16 -> (codes uint8 [rows, K],
    scale float32 [rows])."""
    _cuda(x)
    if x.dim() != 2:
        raise ValueError("x must be [rows, K]")
    q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    sc = torch.empty(x.shape[0], dtype=torch.float32, device=x.device)
    _check(lib().rf_rowquant_e4m3(_ptr(x), x.shape[0], x.shape[1], _ptr(q), _ptr(sc), _dt(x),
                                  _stream()))
    return q, sc


def fp8_gemm(a, sa, w, sw, out=None):
    """rf_fp8_gemm: codes a [M, K], w [N, K] (uint8), scales sa [M], sw [N]
    -> C bf16 [M, N]."""
    _cuda(a, sa, w, sw)
    M, K = a.shape
    N = w.shape[0]
    if w.shape[1] != K or a.dtype != torch.uint8 or w.dtype != torch.uint8:
        raise ValueError("a [M, K] and w [N, K] must be uint8 codes")
    c = torch.empty(M, N, dtype=torch.bfloat16, device=a.device) if out is None else out
    _cuda(c)
    _check(lib().rf_fp8_gemm(_ptr(a), _ptr(sa), _ptr(w), _ptr(sw), _ptr(c), M, N, K, _stream()))
    return c


def mla_decode(q, kv, nsplit, scale, workspace=None, out=None, lse=None):
    """rf_mla_decode: q [B, 128, 576], kv [B, Sk, 576] bf16 -> (o [B, 128, 512]
    bf16, lse [B, 128] float32)."""
    _cuda(q, kv)
    B, Sk = kv.shape[0], kv.shape[1]
    if q.shape != (B, 128, 576) or kv.shape[2] != 576:
        raise ValueError("q must be [B, 128, 576] and kv [B, Sk, 576]")
    o = torch.empty(B, 128, 512, dtype=torch.bfloat16, device=q.device) if out is None else out
    if lse is None:
        lse = torch.empty(B, 128, dtype=torch.float32, device=q.device)
    nbytes = int(lib().rf_mla_decode_workspace_bytes(B, nsplit))
    ws = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=q.device) \
        if workspace is None else workspace
    _cuda(o, lse, ws)
    _check(lib().rf_mla_decode(_ptr(q), _ptr(kv), _ptr(o), _ptr(lse), B, Sk, float(scale),
                               int(nsplit), _ptr(ws), ws.numel() * ws.element_size(), _stream()))
    return o, lse


def attn_fwd(q, k, v, scale=None, causal=False, blockmask=None, out=None, lse=None,
             with_lse=True, kernel="block"):
    """rf_attn_fwd (kernel "block"), rf_attn_fwd_rowwise ("row"), or the one
    rf_attn_choose_kernel picks ("auto"): q [B,H,Sq,d], k/v [B,Hkv,Sk,d] ->
    (o, lse or None)."""
    _cuda(q, k, v)
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if kernel == "auto":
        counts = selector_counts(B, H, Sq, Sk, causal, blockmask, q.device)
        kernel = "row" if choose_kernel(B, H, Sq, Sk, d, *counts, device=q.device) == \
            RF_KERNEL_ROWWISE else "block"
    if kernel not in ("block", "row"):
        raise ValueError("kernel must be 'block', 'row' or 'auto'")
    o = torch.empty_like(q) if out is None else out
    if lse is None and with_lse:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    _cuda(o, lse)
    bm = None
    if blockmask is not None:
        # the tensor-core kernel takes its work in the mask's order (long
        # items first); the other kernels ignore the field
        order = blockmask.cta_order(B, H, Sq) if kernel == "block" and Sq > 0 else None
        bm = ctypes.byref(blockmask.as_struct(order))
    fn = lib().rf_attn_fwd if kernel == "block" else lib().rf_attn_fwd_rowwise
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Sq, Sk, d, float(scale),
              1 if causal else 0, bm, _dt(q), _stream()))
    return o, lse


def attn_fwd_rowwise(q, k, v, scale=None, causal=False, blockmask=None, out=None, lse=None,
                     with_lse=True):
    """rf_attn_fwd_rowwise (STOF's row-wise kernel); arguments as attn_fwd."""
    return attn_fwd(q, k, v, scale, causal, blockmask, out, lse, with_lse, kernel="row")


def choose_kernel(B, H, Sq, Sk, d, listed_tiles, partial_tiles, visible_pairs, num_sms=None,
                  device=None):
    """rf_attn_choose_kernel: RF_KERNEL_BLOCKWISE or RF_KERNEL_ROWWISE."""
    if num_sms is None:
        num_sms = _num_sms(device)
    r = lib().rf_attn_choose_kernel(B, H, Sq, Sk, d, int(listed_tiles), int(partial_tiles),
                                    int(visible_pairs), int(num_sms))
    if r < 0:
        raise ValueError("rf_attn_choose_kernel: invalid arguments")
    return r


def estimate_us(B, H, Sq, Sk, d, listed_tiles, partial_tiles, visible_pairs, num_sms=None,
                device=None):
    """rf_attn_estimate_us: (block-wise, row-wise) model times in microseconds."""
    if num_sms is None:
        num_sms = _num_sms(device)
    b, r = ctypes.c_double(), ctypes.c_double()
    _check(lib().rf_attn_estimate_us(B, H, Sq, Sk, d, int(listed_tiles), int(partial_tiles),
                                     int(visible_pairs), int(num_sms), ctypes.byref(b),
                                     ctypes.byref(r)))
    return b.value, r.value


def _num_sms(device):
    if torch.cuda.is_available():
        dev = torch.cuda.current_device() if device is None else torch.device(device).index or 0
        return torch.cuda.get_device_properties(dev).multi_processor_count
    return 152


def selector_counts(B, H, Sq, Sk, causal, blockmask=None, device=None):
    """rf_blockmask_counts: (listed_tiles, partial_tiles, visible_pairs) over
    all B*H heads, the selector's inputs, counted on the device from the tile
    lists (dense when blockmask is None); waits for the three numbers."""
    dev = blockmask.row_ptr.device if blockmask is not None else (
        torch.device("cuda", torch.cuda.current_device()) if device is None else device)
    counts = torch.empty(3, dtype=torch.int64, device=dev)
    bm = ctypes.byref(blockmask.as_struct()) if blockmask is not None else None
    with torch.cuda.device(dev):
        _check(lib().rf_blockmask_counts(bm, B, H, Sq, Sk, 1 if causal else 0, _ptr(counts),
                                         _stream()))
        listed, partial, pairs = (int(x) for x in counts.cpu().tolist())
    return listed, partial, pairs


def attn_fwd_host_workspace_bytes(B, H, Hkv, Sq, Sk, d, dtype=torch.bfloat16):
    return int(lib().rf_attn_fwd_host_workspace_bytes(
        B, H, Hkv, Sq, Sk, d, RF_F32 if dtype == torch.float32 else RF_BF16))


def attn_fwd_host(q, k, v, scale=None, causal=False, blockmask=None, out=None, lse=None,
                  with_lse=True, workspace=None, device=None):
    """rf_attn_fwd_host: q [B,H,Sq,d], k/v [B,Hkv,Sk,d] in HOST memory (pinned for
    overlap) -> (o, lse) in host memory; copies and kernels pipelined by chunks.
    The call is asynchronous on the current stream of `device`."""
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous host tensors")
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    pin = q.is_pinned()
    o = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin) if out is None else out
    if lse is None and with_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, pin_memory=pin)
    nbytes = attn_fwd_host_workspace_bytes(B, H, Hkv, Sq, Sk, d, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(1, nbytes), dtype=torch.uint8, device=dev)
    _cuda(workspace)
    bm = ctypes.byref(blockmask.as_struct()) if blockmask is not None else None
    with torch.cuda.device(dev):
        _check(lib().rf_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv,
                                      Sq, Sk, d, float(scale), 1 if causal else 0, bm, _dt(q),
                                      _ptr(workspace), workspace.numel(), _stream()))
    return o, lse


def decode_workspace_bytes(B, H, nsplit, d):
    return int(lib().rf_decode_workspace_bytes(B, H, nsplit, d))


def attn_decode_splitk(q, k, v, nsplit, scale=None, workspace=None, out=None, lse=None):
    """rf_attn_decode_splitk: q [B,H,1,d], k/v [B,Hkv,Sk,d] -> (o, lse)."""
    _cuda(q, k, v)
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = decode_workspace_bytes(B, H, nsplit, d)
    if workspace is None:
        workspace = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=q.device)
    o = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    _cuda(workspace, o, lse)
    _check(lib().rf_attn_decode_splitk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv,
                                       Sk, d, float(scale), nsplit, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _dt(q),
                                       _stream()))
    return o, lse


def attn_decode_splitk_noalloc(q, k, v, nsplit, scale=None, out=None, lse=None):
    """rf_attn_decode_splitk_noalloc: the split-K decode with the library's own
    fixed 16 MiB device workspace (for callers that cannot allocate; calls on
    one device share that workspace and must not overlap on the GPU)."""
    _cuda(q, k, v)
    B, H, Sq, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    _cuda(o, lse)
    _check(lib().rf_attn_decode_splitk_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B,
                                               H, Hkv, Sk, d, float(scale), nsplit, _dt(q),
                                               _stream()))
    return o, lse


def attn_decode_partials(q, k, v, nsplit, scale=None, workspace=None):
    """rf_attn_decode_partials: q [B,H,1,d], k/v [B,Hkv,Sk,d] bf16 -> (o_part
    float32 [B*H, nsplit, d], lse_part float32 [B*H, nsplit]), views of the
    workspace."""
    _cuda(q, k, v)
    B, H, _, d = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nbytes = decode_workspace_bytes(B, H, nsplit, d)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device) \
        if workspace is None else workspace
    _cuda(ws)
    _check(lib().rf_attn_decode_partials(_ptr(q), _ptr(k), _ptr(v), _ptr(ws),
                                         ws.numel() * ws.element_size(), B, H, Hkv, Sk, d,
                                         float(scale), int(nsplit), _dt(q), _stream()))
    n = B * H * nsplit
    return ws[:n * d].view(B * H, nsplit, d), ws[n * d:n * d + n].view(B * H, nsplit)


def splitk_merge(o_part, lse_part, out_dtype=torch.bfloat16):
    """rf_splitk_merge: o_part [rows, nsplit, d] f32, lse_part [rows, nsplit] f32.

    Contiguous partials go to rf_splitk_merge; strided views (for instance
    ``gathered.permute(1, 0, 2)`` of split-major [nsplit, rows, d] partials,
    with d contiguous) go to rf_splitk_merge_strided with their strides."""
    for t in (o_part, lse_part):
        if not t.is_cuda or t.dtype != torch.float32:
            raise ValueError("partials must be float32 CUDA tensors")
    rows, nsplit, d = o_part.shape
    if lse_part.shape != (rows, nsplit):
        raise ValueError("lse_part must be [rows, nsplit]")
    o = torch.empty(rows, d, dtype=out_dtype, device=o_part.device)
    lse = torch.empty(rows, dtype=torch.float32, device=o_part.device)
    out_dt = RF_F32 if out_dtype == torch.float32 else RF_BF16
    if o_part.is_contiguous() and lse_part.is_contiguous():
        _check(lib().rf_splitk_merge(_ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), rows,
                                     nsplit, d, out_dt, _stream()))
    else:
        if o_part.stride(2) != 1:
            raise ValueError("o_part's last dimension must be contiguous")
        _check(lib().rf_splitk_merge_strided(
            _ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), rows, nsplit, d, o_part.stride(1),
            o_part.stride(0), lse_part.stride(1), lse_part.stride(0), out_dt, _stream()))
    return o, lse


def set_debug_visited(buf):
    """Record visited tiles of later attn_fwd calls on this thread into a uint8
    CUDA tensor (None turns it off)."""
    if buf is None:
        _check(lib().rf_debug_set_visited(None, 0))
    else:
        _cuda(buf)
        _check(lib().rf_debug_set_visited(_ptr(buf), buf.numel()))


def inject_fault(site):
    """Test aid: later calls on this thread skip one step at ``site`` so that
    a bounded device wait runs out (rf_debug_inject_fault); 0 turns it off."""
    _check(lib().rf_debug_inject_fault(int(site)))


def device_status():
    """Synchronise the current stream; return the device status code (0 = none)
    and clear it. Raises RFError for a nonzero code."""
    code = ctypes.c_int(0)
    st = lib().rf_device_status(_stream(), ctypes.byref(code))
    if st != RF_OK:
        raise RFError(st, lib().rf_last_error().decode(errors="replace"))
    return code.value
