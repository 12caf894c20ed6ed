"""Thin Python binding of ``libpi.so`` (the C ABI declared in ``include/pi.h``).

Argument marshalling only: torch CUDA tensors in, device pointers and the
current CUDA stream out; every step of the decode path runs in the library's
kernels.  The functions carry the C names.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

from .build import LIB

PI_OK, PI_ERR_INVALID_ARG, PI_ERR_UNSUPPORTED, PI_ERR_CUDA, PI_ERR_TIMEOUT, PI_ERR_WORKSPACE = range(6)
PI_W_F16, PI_W_INT4_G32 = 0, 1


class pi_layer_desc(C.Structure):
    _fields_ = [("d", C.c_int), ("ffn", C.c_int), ("rank", C.c_int), ("batch", C.c_int),
                ("wdtype", C.c_int), ("gated", C.c_int)]


class pi_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w1", "w1_scales", "b1", "wu", "w2t", "w2t_scales", "b2",
                                          "p1", "p2", "table")]


class pi_workspace_layout_t(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in ("mask", "idx", "count", "h", "total")]


class pi_cold_tier(C.Structure):
    _fields_ = [("n_hot", C.c_int)] + [(n, C.c_void_p) for n in ("w1", "w1_scales", "wu", "w2t", "w2t_scales")]


class pi_stack_plan_t(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("fused", "ctas", "pred_in_smem", "p2_ring_slots", "fc_row_slots",
                                       "smem_bytes")]


class pi_attn_desc(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("d", "heads", "kv_heads", "head_dim", "rank", "batch", "max_seq")]


class pi_attn_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("wqkv", "bqkv", "wot", "bo", "p1", "p2", "bp")]


class PiError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


_lib = None

EXPORTS = ("pi_workspace_bytes", "pi_workspace_layout", "pi_predict", "pi_compact", "pi_sparse_fc1",
           "pi_sparse_fc2", "pi_ffn_layer", "pi_rmsnorm_half", "pi_status_string",
           "pi_last_device_status", "pi_launches_per_layer", "pi_ffn_stack", "pi_debug_wait_timeout",
           "pi_sparse_fc2_noalloc", "pi_stack_plan", "pi_stack_plan_for", "pi_debug_set_wait_timeout",
           "pi_sparse_fc1_tiered", "pi_sparse_fc2_tiered", "pi_ffn_layer_tiered", "pi_attn_workspace_bytes",
           "pi_attn_heads")


def library_path() -> str:
    return LIB


def lib(path: Optional[str] = None):
    """Load ``libpi.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libpi.so not built ({p}); run __graft_entry__.build() or "
                           "python -m activation_sparse_ffn_layer_gb300.build")
    L = C.CDLL(p)
    P, I, Fl, S = C.c_void_p, C.c_int, C.c_float, C.c_size_t
    D = C.POINTER(pi_layer_desc)
    Wt = C.POINTER(pi_layer_weights)
    sig = {
        "pi_workspace_bytes": (S, [D]),
        "pi_workspace_layout": (I, [D, C.POINTER(pi_workspace_layout_t)]),
        "pi_predict": (I, [D, P, P, P, P, Fl, P, P, S, P]),
        "pi_compact": (I, [D, P, P, P, P, P, P]),
        "pi_sparse_fc1": (I, [D, P, Wt, P, P, P, P, P, S, P]),
        "pi_sparse_fc2": (I, [D, P, P, P, Wt, P, P, S, P]),
        "pi_ffn_layer": (I, [D, P, Wt, Fl, P, S, P, P]),
        "pi_rmsnorm_half": (I, [I, I, P, Fl, P, P]),
        "pi_status_string": (C.c_char_p, [I]),
        "pi_last_device_status": (I, [P]),
        "pi_launches_per_layer": (I, [D]),
        "pi_ffn_stack": (I, [D, I, C.POINTER(pi_layer_weights), P, P, Fl, Fl, P, S, P, P, P, P]),
        "pi_debug_wait_timeout": (I, [C.c_longlong, P]),
        "pi_sparse_fc2_noalloc": (I, [D, P, P, P, Wt, P, P]),
        "pi_stack_plan": (I, [D, I, P, C.POINTER(pi_stack_plan_t)]),
        "pi_stack_plan_for": (I, [D, I, P, I, C.POINTER(pi_stack_plan_t)]),
        "pi_debug_set_wait_timeout": (I, [C.c_longlong]),
        "pi_sparse_fc1_tiered": (I, [D, P, Wt, C.POINTER(pi_cold_tier), P, P, P, P, P]),
        "pi_sparse_fc2_tiered": (I, [D, P, P, P, Wt, C.POINTER(pi_cold_tier), P, P, S, P]),
        "pi_ffn_layer_tiered": (I, [D, P, Wt, C.POINTER(pi_cold_tier), Fl, P, S, P, P]),
        "pi_attn_workspace_bytes": (S, [C.POINTER(pi_attn_desc)]),
        "pi_attn_heads": (I, [C.POINTER(pi_attn_desc), P, C.POINTER(pi_attn_weights), P, P, P, Fl, P, P, P, S,
                              P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = L
    return L


# ------------------------------------------------------------------ marshalling

def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn: str, st: int):
    if st != PI_OK:
        raise PiError(fn, st, lib().pi_status_string(st).decode())


def desc_of(d: int, ffn: int, rank: int, batch: int = 1, int4: bool = False, gated: bool = False) -> pi_layer_desc:
    return pi_layer_desc(d, ffn, rank, batch, PI_W_INT4_G32 if int4 else PI_W_F16, 1 if gated else 0)


def layer_desc(w, batch: int = 1) -> pi_layer_desc:
    return desc_of(w.d, w.F, w.r, batch, w.int4, w.gated)


def weights_struct(w) -> pi_layer_weights:
    """A pi_layer_weights over a layer's device tensors (keep `w` alive)."""
    s = pi_layer_weights()
    if w.int4:
        s.w1, s.w1_scales = _ptr(w.w1_q), _ptr(w.w1_s)
        s.w2t, s.w2t_scales = _ptr(w.w2t_q), _ptr(w.w2t_s)
    else:
        s.w1, s.w2t = _ptr(w.w1), _ptr(w.w2t)
    s.b1, s.b2, s.p1, s.p2, s.table = _ptr(w.b1), _ptr(w.b2), _ptr(w.p1), _ptr(w.p2), _ptr(w.table)
    if w.gated:
        s.wu = _ptr(w.wu)
    return s


# ------------------------------------------------------------- the C entry points

def pi_workspace_bytes(desc: pi_layer_desc) -> int:
    return int(lib().pi_workspace_bytes(C.byref(desc)))


def pi_workspace_layout(desc: pi_layer_desc) -> pi_workspace_layout_t:
    out = pi_workspace_layout_t()
    _check("pi_workspace_layout", lib().pi_workspace_layout(C.byref(desc), C.byref(out)))
    return out


def pi_predict(desc, x, p1, p2, bpred, tau: float, mask, workspace):
    _check("pi_predict", lib().pi_predict(C.byref(desc), _ptr(x), _ptr(p1), _ptr(p2), _ptr(bpred),
                                          float(tau), _ptr(mask), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream()))


def pi_compact(desc, mask, table, idx, orig_idx, d_count):
    _check("pi_compact", lib().pi_compact(C.byref(desc), _ptr(mask), _ptr(table), _ptr(idx), _ptr(orig_idx),
                                          _ptr(d_count), _stream()))


def pi_sparse_fc1(desc, x, wstruct, idx, d_count, mask, h, workspace):
    _check("pi_sparse_fc1", lib().pi_sparse_fc1(C.byref(desc), _ptr(x), C.byref(wstruct), _ptr(idx),
                                                _ptr(d_count), _ptr(mask), _ptr(h), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream()))


def pi_sparse_fc2(desc, h, idx, d_count, wstruct, y, workspace):
    _check("pi_sparse_fc2", lib().pi_sparse_fc2(C.byref(desc), _ptr(h), _ptr(idx), _ptr(d_count),
                                                C.byref(wstruct), _ptr(y), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream()))


def pi_sparse_fc2_noalloc(desc, h, idx, d_count, wstruct, y):
    """pi_sparse_fc2 without a workspace: for callers that cannot allocate
    device memory (the partial sums live in a fixed array inside the library;
    calls must not overlap on the GPU)."""
    _check("pi_sparse_fc2_noalloc", lib().pi_sparse_fc2_noalloc(C.byref(desc), _ptr(h), _ptr(idx), _ptr(d_count),
                                                                C.byref(wstruct), _ptr(y), _stream()))


def pi_ffn_layer(desc, x, wstruct, tau: float, workspace, y):
    _check("pi_ffn_layer", lib().pi_ffn_layer(C.byref(desc), _ptr(x), C.byref(wstruct), float(tau),
                                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              _ptr(y), _stream()))


def pi_ffn_stack(desc, wstructs, ranks, x, tau: float, eps: float, workspace, y, x_trace=None,
                 layer_counts=None):
    """`wstructs`: a ctypes array of pi_layer_weights (see weights_array);
    `ranks`: a ctypes int array or None; `layer_counts`: int32 [L, 2] or None."""
    n = len(wstructs)
    _check("pi_ffn_stack", lib().pi_ffn_stack(C.byref(desc), n, wstructs, ranks, _ptr(x), float(tau), float(eps),
                                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              _ptr(y), _ptr(x_trace), _ptr(layer_counts), _stream()))


def weights_array(layers):
    """A ctypes array of pi_layer_weights over a list of layers (keep them alive)."""
    arr = (pi_layer_weights * len(layers))()
    for i, w in enumerate(layers):
        arr[i] = weights_struct(w)
    return arr


def ranks_array(layers):
    return (C.c_int * len(layers))(*[int(w.r) for w in layers])


def _addr(t):
    """Address of a tensor for the C ABI: device memory, or host memory the
    GPU can address (pinned)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("expected a CUDA tensor or pinned host memory")
    return C.c_void_p(t.data_ptr())


def cold_tier(n_hot: int, w1=None, w1_scales=None, wu=None, w2t=None, w2t_scales=None) -> pi_cold_tier:
    """A pi_cold_tier over tensors in device or pinned host memory (keep them alive)."""
    s = pi_cold_tier()
    s.n_hot = int(n_hot)
    s.w1, s.w1_scales, s.wu = _addr(w1), _addr(w1_scales), _addr(wu)
    s.w2t, s.w2t_scales = _addr(w2t), _addr(w2t_scales)
    return s


def pi_sparse_fc1_tiered(desc, x, wstruct, cold, idx, d_count, mask, h):
    _check("pi_sparse_fc1_tiered", lib().pi_sparse_fc1_tiered(C.byref(desc), _ptr(x), C.byref(wstruct), C.byref(cold),
                                                              _ptr(idx), _ptr(d_count), _ptr(mask), _ptr(h),
                                                              _stream()))


def pi_sparse_fc2_tiered(desc, h, idx, d_count, wstruct, cold, y, workspace):
    _check("pi_sparse_fc2_tiered", lib().pi_sparse_fc2_tiered(C.byref(desc), _ptr(h), _ptr(idx), _ptr(d_count),
                                                              C.byref(wstruct), C.byref(cold), _ptr(y),
                                                              _ptr(workspace),
                                                              workspace.numel() * workspace.element_size(),
                                                              _stream()))


def pi_ffn_layer_tiered(desc, x, wstruct, cold, tau: float, workspace, y):
    _check("pi_ffn_layer_tiered", lib().pi_ffn_layer_tiered(C.byref(desc), _ptr(x), C.byref(wstruct), C.byref(cold),
                                                            float(tau), _ptr(workspace),
                                                            workspace.numel() * workspace.element_size(), _ptr(y),
                                                            _stream()))


def pi_stack_plan(desc, n_layers: int, ranks=None) -> pi_stack_plan_t:
    """How a pi_ffn_stack step of `n_layers` layers runs on the current device."""
    out = pi_stack_plan_t()
    _check("pi_stack_plan", lib().pi_stack_plan(C.byref(desc), int(n_layers), ranks, C.byref(out)))
    return out


def pi_stack_plan_for(desc, n_layers: int, sm_count: int, ranks=None) -> pi_stack_plan_t:
    """The same plan for a device with `sm_count` SMs (host only, no device)."""
    out = pi_stack_plan_t()
    _check("pi_stack_plan_for", lib().pi_stack_plan_for(C.byref(desc), int(n_layers), ranks, int(sm_count),
                                                        C.byref(out)))
    return out


def pi_debug_set_wait_timeout(timeout_ns: int):
    _check("pi_debug_set_wait_timeout", lib().pi_debug_set_wait_timeout(int(timeout_ns)))


def pi_debug_wait_timeout(timeout_ns: int):
    _check("pi_debug_wait_timeout", lib().pi_debug_wait_timeout(int(timeout_ns), _stream()))


def pi_rmsnorm_half(d: int, batch: int, y, eps: float, x_out):
    _check("pi_rmsnorm_half", lib().pi_rmsnorm_half(int(d), int(batch), _ptr(y), float(eps), _ptr(x_out),
                                                    _stream()))


def pi_status_string(status: int) -> str:
    return lib().pi_status_string(int(status)).decode()


def pi_launches_per_layer(desc) -> int:
    return int(lib().pi_launches_per_layer(C.byref(desc)))


def pi_last_device_status() -> int:
    return int(lib().pi_last_device_status(_stream()))


# ------------------------------------------------------- head-sparse attention

def attn_desc_of(d: int, heads: int, kv_heads: int, head_dim: int, rank: int, batch: int = 1,
                 max_seq: int = 1024) -> pi_attn_desc:
    return pi_attn_desc(d, heads, kv_heads, head_dim, rank, batch, max_seq)


def attn_desc(w, batch: int = 1, max_seq: int = 1024) -> pi_attn_desc:
    return attn_desc_of(w.d, w.H, w.KVH, w.dh, w.r, batch, max_seq)


def attn_weights_struct(w) -> pi_attn_weights:
    """A pi_attn_weights over an attention block's device tensors (keep `w` alive)."""
    s = pi_attn_weights()
    s.wqkv, s.bqkv, s.wot, s.bo = _ptr(w.wqkv), _ptr(w.bqkv), _ptr(w.wot), _ptr(w.bo)
    s.p1, s.p2, s.bp = _ptr(w.p1), _ptr(w.p2), _ptr(w.bp)
    return s


def pi_attn_workspace_bytes(desc: pi_attn_desc) -> int:
    return int(lib().pi_attn_workspace_bytes(C.byref(desc)))


def pi_attn_heads(desc, x, wstruct, kcache, vcache, pos, tau: float, head_mask, y, workspace):
    _check("pi_attn_heads", lib().pi_attn_heads(C.byref(desc), _ptr(x), C.byref(wstruct), _ptr(kcache),
                                                _ptr(vcache), _ptr(pos), float(tau), _ptr(head_mask), _ptr(y),
                                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                _stream()))
