"""The C-ABI library loads, exports every entry point that include/pi.h
declares, and rejects bad arguments on the host without launching anything."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pi.h")).read()
    return sorted(set(re.findall(r"PI_API\s+[\w\s\*]+?\b(pi_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def P():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_ffn_layer_gb300 as P
    return P


def test_every_declared_symbol_is_exported(P):
    names = _declared()
    assert len(names) >= 10, names
    raw = C.CDLL(P.library_path())
    for n in names:
        assert hasattr(raw, n), f"{n} declared in pi.h but not exported"
    assert set(names) == set(P.binding.EXPORTS) | set(n for n in names if n not in P.binding.EXPORTS)
    for n in P.binding.EXPORTS:
        assert n in names, f"binding wraps {n} which pi.h does not declare"


def test_status_strings(P):
    for st in range(6):
        assert P.pi_status_string(st)


def test_host_validation_without_launch(P):
    L = P.lib()
    ok = P.desc_of(256, 1000, 32, 1)
    assert P.pi_workspace_bytes(ok) > 0
    for bad in (P.desc_of(250, 1000, 32, 1), P.desc_of(256, 0, 32, 1), P.desc_of(256, 1000, 30, 1),
                P.desc_of(256, 1000, 32, 0), P.desc_of(256, 1000, 32, 33), P.desc_of(48, 64, 8, 1, int4=True)):
        assert P.pi_workspace_bytes(bad) == 0
        assert L.pi_ffn_layer(C.byref(bad), None, None, -0.05, None, 0, None, None) == 1
    # valid descriptor, missing pointers: rejected before any launch
    assert L.pi_ffn_layer(C.byref(ok), None, None, -0.05, None, 0, None, None) == 1
    assert L.pi_compact(C.byref(ok), None, None, None, None, None, None) == 1
    assert L.pi_ffn_layer(None, None, None, 0.0, None, 0, None, None) == 1
    assert L.pi_rmsnorm_half(0, 1, None, 1e-6, None, None) == 1


def test_attention_descriptor_validation_without_launch(P):
    """pi_attn_workspace_bytes sizes only valid blocks; pi_attn_heads rejects a
    bad descriptor or missing pointers on the host (status 1), a missing
    workspace with status 5, and launches nothing."""
    L = P.lib()
    ok = P.attn_desc_of(256, 8, 2, 64, 16, 2, 64)
    assert P.pi_attn_workspace_bytes(ok) > 0
    bad = [
        P.attn_desc_of(250, 8, 2, 64, 16, 2, 64),     # d not a multiple of 8
        P.attn_desc_of(256, 8, 3, 64, 16, 2, 64),     # heads not a multiple of the KV heads
        P.attn_desc_of(256, 8, 2, 96, 16, 2, 64),     # head_dim other than 64 / 128
        P.attn_desc_of(256, 8, 2, 64, 12, 2, 64),     # rank not a multiple of 8
        P.attn_desc_of(256, 8, 2, 64, 16, 33, 64),    # batch above 32
        P.attn_desc_of(256, 8, 2, 64, 16, 2, 0),      # no cache positions
        P.attn_desc_of(256, 0, 1, 64, 16, 2, 64),     # no heads
    ]
    for b in bad:
        assert P.pi_attn_workspace_bytes(b) == 0
        assert L.pi_attn_heads(C.byref(b), None, None, None, None, None, 0.0, None, None, None, 0, None) == 1
    w = P.binding.pi_attn_weights()
    assert L.pi_attn_heads(C.byref(ok), None, C.byref(w), None, None, None, 0.0, None, None, None, 0, None) == 1
    assert L.pi_attn_heads(None, None, None, None, None, None, 0.0, None, None, None, 0, None) == 1
    # every pointer present and 16-byte aligned (never dereferenced: the
    # workspace check comes first), the workspace missing or too small
    fake = C.c_void_p(1 << 20)
    wf = P.binding.pi_attn_weights(*([1 << 20] * 7))
    need = P.pi_attn_workspace_bytes(ok)
    for ws, nbytes in ((None, need), (fake, need - 16)):
        assert L.pi_attn_heads(C.byref(ok), fake, C.byref(wf), fake, fake, fake, 0.0, fake, fake, ws, nbytes,
                               None) == 5
