"""CPU oracle of the neuron-aware sparse FFN decode path (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The CUDA library never imports, links or
calls this package, and this package never touches the CUDA library.

This module marshals numpy / torch-CPU arrays into ``liboracle.so`` (built from
``oracle.c`` on first use).  All arithmetic is in the C file; see its header
for the passages each function follows and the readings taken where the pages
are silent.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build as _build

_lib = None


class _Mat(C.Structure):
    _fields_ = [("kind", C.c_int), ("f16", C.c_void_p), ("q", C.c_void_p), ("scales", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = _build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.oracle_half_to_double.restype = C.c_double
        L.oracle_half_to_double.argtypes = [C.c_uint16]
        L.oracle_double_to_half.restype = C.c_uint16
        L.oracle_double_to_half.argtypes = [C.c_double]
        L.oracle_decode_row.argtypes = [P, C.c_int, C.c_long, P]
        L.oracle_predict.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P, P, C.c_float, C.c_double,
                                     P, P, P, P]
        L.oracle_compact.argtypes = [C.c_int, P, P, P, P, P]
        L.oracle_mask_union.argtypes = [C.c_int, C.c_int, P, P]
        L.oracle_fc1.argtypes = [C.c_int, C.c_int, P, P, P, P, P, C.c_int, P]
        L.oracle_fc2.argtypes = [C.c_int, P, P, P, P, C.c_int, P]
        L.oracle_ffn_masked.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P, P, P, P, P, P, P]
        L.oracle_ffn_dense.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P, P, P, P, P]
        L.oracle_rmsnorm_half.argtypes = [C.c_int, P, C.c_double, C.c_double, P, P, P]
        L.oracle_attn_heads.argtypes = [C.c_int] * 6 + [P] * 10 + [C.c_double, P, P]
        L.oracle_set_threads.argtypes = [C.c_int]
        L.oracle_threads.restype = C.c_int
        for name in ("oracle_decode_row", "oracle_predict", "oracle_compact", "oracle_mask_union",
                     "oracle_fc1", "oracle_fc2", "oracle_ffn_masked", "oracle_ffn_dense",
                     "oracle_rmsnorm_half", "oracle_attn_heads"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


# ------------------------------------------------------------------ helpers

def _np(a, dtype):
    """A C-contiguous numpy array of `dtype` (fp16 data travels as uint16 bits)."""
    if hasattr(a, "detach"):                       # torch tensor
        a = a.detach().cpu()
        if str(a.dtype) == "torch.float16":
            a = a.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        else:
            a = a.contiguous().numpy()
    a = np.asarray(a)
    if dtype == np.uint16 and a.dtype == np.float16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what} rejected its arguments (code {rc})")


class Matrix:
    """A weight matrix with rows of ``d`` elements: fp16 rows, or INT4 group-32
    codes + fp16 scales."""

    def __init__(self, f16=None, q=None, scales=None):
        self.f16 = None if f16 is None else _np(f16, np.uint16)
        self.q = None if q is None else _np(q, np.uint8)
        self.scales = None if scales is None else _np(scales, np.uint16)
        self._s = _Mat(0 if self.f16 is not None else 1, _p(self.f16), _p(self.q), _p(self.scales))

    @property
    def ref(self):
        return C.byref(self._s)


class HostLayer:
    """Host copies of one layer in the oracle's format (bits, not values)."""

    def __init__(self, w):
        self.d, self.F, self.r = int(w.d), int(w.F), int(w.r)
        self.gated = bool(w.gated)
        if getattr(w, "int4", False):
            self.w1 = Matrix(q=w.w1_q, scales=w.w1_s)
            self.w2t = Matrix(q=w.w2t_q, scales=w.w2t_s)
        else:
            self.w1 = Matrix(f16=w.w1)
            self.w2t = Matrix(f16=w.w2t)
        self.wu = Matrix(f16=w.wu) if self.gated else None
        self.b1 = _np(w.b1, np.uint16)
        self.b2 = _np(w.b2, np.uint16)
        self.p1 = _np(w.p1, np.uint16)
        self.p2 = _np(w.p2, np.uint16)
        self.table = _np(w.table, np.int32)


def host_layer(w) -> HostLayer:
    return w if isinstance(w, HostLayer) else HostLayer(w)


# ---------------------------------------------------------------- numbers

def half_to_double(bits) -> np.ndarray:
    b = _np(bits, np.uint16).ravel()
    f = lib().oracle_half_to_double
    return np.array([f(int(v)) for v in b], dtype=np.float64)


def double_to_half(vals) -> np.ndarray:
    v = np.ascontiguousarray(vals, dtype=np.float64).ravel()
    f = lib().oracle_double_to_half
    return np.array([f(float(t)) for t in v], dtype=np.uint16)


def decode_row(mat: Matrix, d: int, row: int) -> np.ndarray:
    out = np.empty(d, dtype=np.float64)
    _check(lib().oracle_decode_row(mat.ref, d, row, _p(out)), "oracle_decode_row")
    return out


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def threads() -> int:
    return int(lib().oracle_threads())


# ---------------------------------------------------------------- the path

FP32_UNIT_ROUNDOFF = 2.0 ** -24


def predict(x, w, tau: float, unit_roundoff: float = FP32_UNIT_ROUNDOFF):
    """Predictor for one token: returns dict(u, s, band, mask)."""
    L = host_layer(w)
    xb = _np(x, np.uint16)
    u = np.empty(L.r, np.float64)
    s = np.empty(L.F, np.float64)
    band = np.empty(L.F, np.float64)
    mask = np.empty((L.F + 31) // 32, np.uint32)
    _check(lib().oracle_predict(L.d, L.F, L.r, _p(xb), _p(L.p1), _p(L.p2), _p(L.b1), float(tau),
                                float(unit_roundoff), _p(u), _p(s), _p(band), _p(mask)),
           "oracle_predict")
    return dict(u=u, s=s, band=band, mask=mask)


def compact(mask, F: int, table=None):
    """Returns (idx, orig, count) with idx/orig cut to `count` entries."""
    m = _np(mask, np.uint32)
    idx = np.empty(max(F, 1), np.int32)
    orig = np.empty(max(F, 1), np.int32)
    tb = None if table is None else _np(table, np.int32)
    cnt = np.zeros(1, np.int32)
    _check(lib().oracle_compact(F, _p(m), _p(tb), _p(idx), _p(orig) if tb is not None else None,
                                _p(cnt)), "oracle_compact")
    n = int(cnt[0])
    return idx[:n].copy(), (orig[:n].copy() if tb is not None else None), n


def mask_union(masks, F: int):
    m = _np(masks, np.uint32)
    B = m.shape[0]
    out = np.empty((F + 31) // 32, np.uint32)
    _check(lib().oracle_mask_union(B, F, _p(m), _p(out)), "oracle_mask_union")
    return out


def fc1(x, w, idx):
    L = host_layer(w)
    xb = _np(x, np.uint16)
    ix = _np(idx, np.int32)
    h = np.empty(max(ix.size, 1), np.float64)
    _check(lib().oracle_fc1(L.d, int(L.gated), _p(xb), L.w1.ref, _p(L.b1),
                            L.wu.ref if L.gated else None, _p(ix), int(ix.size), _p(h)), "oracle_fc1")
    return h[: ix.size]


def fc2(h, w, idx):
    L = host_layer(w)
    hv = np.ascontiguousarray(h, dtype=np.float64)
    ix = _np(idx, np.int32)
    y = np.empty(L.d, np.float64)
    _check(lib().oracle_fc2(L.d, L.w2t.ref, _p(L.b2), _p(hv), _p(ix), int(ix.size), _p(y)), "oracle_fc2")
    return y


def ffn_masked(x, w, mask):
    L = host_layer(w)
    xb = _np(x, np.uint16)
    m = _np(mask, np.uint32)
    y = np.empty(L.d, np.float64)
    _check(lib().oracle_ffn_masked(L.d, L.F, int(L.gated), _p(xb), L.w1.ref, _p(L.b1),
                                   L.wu.ref if L.gated else None, L.w2t.ref, _p(L.b2), _p(L.table),
                                   _p(m), _p(y)), "oracle_ffn_masked")
    return y


def ffn_dense(x, w):
    L = host_layer(w)
    xb = _np(x, np.uint16)
    y = np.empty(L.d, np.float64)
    _check(lib().oracle_ffn_dense(L.d, L.F, int(L.gated), _p(xb), L.w1.ref, _p(L.b1),
                                  L.wu.ref if L.gated else None, L.w2t.ref, _p(L.b2), _p(y)),
           "oracle_ffn_dense")
    return y


def rmsnorm_half(y, eps: float = 1e-6, unit_roundoff: float = FP32_UNIT_ROUNDOFF):
    """Returns (x_bits uint16, pre-rounding values, band)."""
    yv = np.ascontiguousarray(y, dtype=np.float64).ravel()
    d = yv.size
    xb = np.empty(d, np.uint16)
    pre = np.empty(d, np.float64)
    band = np.empty(d, np.float64)
    _check(lib().oracle_rmsnorm_half(d, _p(yv), float(eps), float(unit_roundoff), _p(xb), _p(pre),
                                     _p(band)), "oracle_rmsnorm_half")
    return xb, pre, band


def layer_step(x, w, tau: float, eps: float = 1e-6):
    """One decode layer as the oracle sees it: predict, compact, masked FFN.
    Returns dict(mask, idx, count, y)."""
    L = host_layer(w)
    pr = predict(x, L, tau)
    idx, _, n = compact(pr["mask"], L.F, L.table)
    y = ffn_masked(x, L, pr["mask"])
    return dict(mask=pr["mask"], s=pr["s"], band=pr["band"], idx=idx, count=n, y=y)


# ------------------------------------------------------- attention heads

def attn_predict(x, p1, p2, bp, tau: float, unit_roundoff: float = FP32_UNIT_ROUNDOFF):
    """Head predictor of one token (oracle_predict with F = number of heads):
    dict(u, s, band, mask)."""
    xb = _np(x, np.uint16)
    P1, P2, BP = _np(p1, np.uint16), _np(p2, np.uint16), _np(bp, np.uint16)
    r, d = P1.shape
    H = P2.shape[0]
    u = np.empty(r, np.float64)
    s = np.empty(H, np.float64)
    band = np.empty(H, np.float64)
    mask = np.empty((H + 31) // 32, np.uint32)
    _check(lib().oracle_predict(d, H, r, _p(xb), _p(P1), _p(P2), _p(BP), float(tau), float(unit_roundoff),
                                _p(u), _p(s), _p(band), _p(mask)), "oracle_predict")
    return dict(u=u, s=s, band=band, mask=mask)


def attn_heads(x, wqkv, bqkv, wot, bo, head_mask, kcache, vcache, pos, H: int, KVH: int, dh: int,
               unit_roundoff: float = FP32_UNIT_ROUNDOFF):
    """One decode token per sequence through the head-sparse attention block.

    x [B, d] fp16; wqkv [(H + 2 KVH) dh, d], bqkv, wot [H dh, d], bo [d] fp16;
    head_mask [B, ceil(H/32)] uint32; kcache, vcache [B, KVH, smax, dh] fp16
    (not modified: updated copies are returned); pos [B] ints.
    Returns dict(y [B, d] float64, o [B, H dh] float64, kcache, vcache as
    uint16 bit arrays with position pos[b] written, kv_pre / kv_band [B, 2 KVH dh]:
    the new keys then values before rounding, and the fp32 evaluation bound)."""
    xb = _np(x, np.uint16)
    if xb.ndim == 1:
        xb = xb[None]
    B, d = xb.shape
    W, Bq, Wo, Bo = _np(wqkv, np.uint16), _np(bqkv, np.uint16), _np(wot, np.uint16), _np(bo, np.uint16)
    m = _np(head_mask, np.uint32).reshape(B, -1)
    kc = _np(kcache, np.uint16).copy()
    vc = _np(vcache, np.uint16).copy()
    smax = kc.shape[-2]
    kc = kc.reshape(B, KVH, smax, dh)
    vc = vc.reshape(B, KVH, smax, dh)
    ps = [int(v) for v in np.asarray(pos).ravel()]
    y = np.empty((B, d), np.float64)
    o = np.empty((B, H * dh), np.float64)
    pre = np.empty((B, 2 * KVH * dh), np.float64)
    band = np.empty((B, 2 * KVH * dh), np.float64)
    for b in range(B):
        kb = np.ascontiguousarray(kc[b])
        vb = np.ascontiguousarray(vc[b])
        xr = np.ascontiguousarray(xb[b])
        mr = np.ascontiguousarray(m[b])
        yr = np.empty(d, np.float64)
        orow = np.empty(H * dh, np.float64)
        pr = np.empty(2 * KVH * dh, np.float64)
        bd = np.empty(2 * KVH * dh, np.float64)
        _check(lib().oracle_attn_heads(d, H, KVH, dh, smax, ps[b], _p(xr), _p(W), _p(Bq), _p(Wo), _p(Bo),
                                       _p(mr), _p(kb), _p(vb), _p(orow), _p(yr), float(unit_roundoff), _p(pr),
                                       _p(bd)), "oracle_attn_heads")
        kc[b], vc[b], y[b], o[b], pre[b], band[b] = kb, vb, yr, orow, pr, bd
    return dict(y=y, o=o, kcache=kc, vcache=vc, kv_pre=pre, kv_band=band)
