"""Parity of the one-launch stack decode step (pi_ffn_stack) against the
oracle, layer by layer, plus determinism and the bounded-wait status path."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close, half_matches, mask_matches

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pi():
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    return P


def _mask_of(P, st):
    lay = P.pi_workspace_layout(st.desc)
    W = (st.layers[0].w.F + 31) // 32
    return st.workspace[lay.mask:lay.mask + 4 * W].view(torch.int32).cpu().numpy().view(np.uint32)


def _check_stack(cfg, L, token=0):
    """Run prefixes of the stack (1..L layers): the workspace then holds layer
    l's mask, y_out is layer l's output and x_trace its inputs."""
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    ws = [make_layer(cfg, l, device=DEV) for l in range(L)]
    hosts = [oracle.host_layer(w.to("cpu")) for w in ws]
    x = make_tokens(cfg, token, 1, device=DEV)
    ambiguous = 0
    full = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    xs_full, y_full = full.step_trace(x)
    for l in range(L):
        st = DecodeStack(ws[: l + 1], batch=1, tau=cfg.tau, eps=cfg.rms_eps)
        xs, y = st.step_trace(x)
        torch.cuda.synchronize()
        # the prefix run and the full run agree on every shared layer input
        for j in range(l + 1):
            assert torch.equal(xs[j], xs_full[j]), f"layer {j} input differs between runs"
        mask = _mask_of(P, st)
        xl = xs[l][0].cpu()
        ambiguous += mask_matches(mask, oracle.predict(xl, hosts[l], cfg.tau), cfg.F, cfg.tau, f"layer {l}")
        yo = oracle.ffn_masked(xl, hosts[l], mask)
        close(y[0].cpu().numpy(), yo, f"{cfg.key} stack layer {l}")
        if l + 1 < L:
            _, pre, band = oracle.rmsnorm_half(y[0].cpu().numpy().astype(np.float64), cfg.rms_eps)
            half_matches(xs_full[l + 1][0].cpu().view(torch.int16).numpy().view(np.uint16), pre, band,
                         f"normalised input of layer {l + 1}")
    close(y_full[0].cpu().numpy(), y[0].cpu().numpy(), "full run vs prefix run", max_abs=0, rel_l2=0)
    return ambiguous


@pytest.mark.parametrize("name,cfg,L", [
    ("c2-small", small(CONFIGS["c2"], d=1024, F=4096, rank=64), 5),
    ("gated-small", small(CONFIGS["c4"], d=1024, F=3000, rank=64), 3),
    ("int4-small", small(CONFIGS["c5"], d=1024, F=4100, rank=128), 3),
    ("ragged", small(CONFIGS["c1"], d=264, F=1001, rank=24), 3),
    # wider than the columns each thread prefetches in registers (tail loop of x)
    ("int4-wide", small(CONFIGS["c5"], d=10240, F=2048, rank=64), 2),
    ("fp16-wide", small(CONFIGS["c4"], d=8192, F=2000, rank=64), 2),
])
def test_stack_layers_match_oracle(name, cfg, L):
    _check_stack(cfg, L)


def test_stack_c2_full_shape_first_layers():
    _check_stack(CONFIGS["c2"], 3)


def test_stack_repeatable_and_epochs_advance():
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    ws = [make_layer(cfg, l, device=DEV) for l in range(4)]
    st = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    xs = make_tokens(cfg, 0, 3, device=DEV)
    outs = []
    for rep in range(3):
        for t in range(3):
            outs.append((t, st.step(xs[t:t + 1]).clone()))
    torch.cuda.synchronize()
    for t in range(3):
        ys = [y for tt, y in outs if tt == t]
        assert all(torch.equal(ys[0], y) for y in ys[1:])
    assert not torch.equal(outs[0][1], outs[1][1])
    assert P.pi_last_device_status() == 0


def test_stack_graph_replay_matches_eager():
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    ws = [make_layer(cfg, l, device=DEV) for l in range(3)]
    st = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    xs = make_tokens(cfg, 0, 4, device=DEV)
    eager = [st.step(xs[t:t + 1]).clone() for t in range(4)]
    st.capture()
    for t in range(4):
        st.x_in.copy_(xs[t:t + 1])
        st.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.y, eager[t])


def test_bounded_wait_times_out_and_context_survives():
    P = _pi()
    assert P.pi_last_device_status() == 0
    P.pi_debug_wait_timeout(2_000_000)          # 2 ms on a word nothing writes
    assert P.pi_last_device_status() == 4       # PI_ERR_TIMEOUT, read once ...
    assert P.pi_last_device_status() == 0       # ... then cleared
    # the context is still usable
    cfg = small(CONFIGS["c1"], d=256, F=1000, rank=32)
    w = make_layer(cfg, 0, device=DEV)
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    st = DecodeStack([w], batch=1, tau=cfg.tau)
    x = make_tokens(cfg, 0, 1, device=DEV)
    y = st.step(x).clone()
    torch.cuda.synchronize()
    close(y[0].cpu().numpy(), oracle.ffn_masked(x[0].cpu(), oracle.host_layer(w.to("cpu")), _mask_of(P, st)),
          "layer after timeout")
    assert P.pi_last_device_status() == 0


def test_layer_counts_match_last_layer_workspace():
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    ws = [make_layer(cfg, l, device=DEV) for l in range(3)]
    st = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    x = make_tokens(cfg, 0, 1, device=DEV)
    cnt = st.step_counts(x).cpu().numpy()
    lay = P.pi_workspace_layout(st.desc)
    n = int(st.workspace[lay.count:lay.count + 4].view(torch.int32).item())
    h = st.workspace[lay.h:lay.h + 4 * n].view(torch.float32).cpu().numpy()
    assert cnt.shape == (3, 2)
    assert cnt[2, 0] == n and cnt[2, 1] == int((h != 0).sum())
    assert np.all(cnt[:, 1] <= cnt[:, 0]) and np.all(cnt[:, 0] > 0)
