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


def _check_stack(cfg, L, token=0, p2_ring=False):
    """Run prefixes of the stack (1..L layers): the workspace then holds layer
    l's mask, y_out is layer l's output and x_trace its inputs.  With p2_ring
    the plan must stream P2 through the ring of 16-row slots."""
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    ws = [make_layer(cfg, l, device=DEV) for l in range(L)]
    hosts = [oracle.host_layer(w.to("cpu")) for w in ws]
    x = make_tokens(cfg, token, 1, device=DEV)
    ambiguous = 0
    full = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    if p2_ring:
        plan = P.pi_stack_plan(full.desc, L, full.ranks)
        assert plan.fused == 1 and plan.pred_in_smem == 0 and plan.p2_ring_slots >= 2, "P2 ring not taken"
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


@pytest.mark.parametrize("name,cfg,L", [
    # rank 1024 over 16390 rows: a block's P2 share (≥ 6 units of 32 KB) does not
    # fit in shared memory, so P2 streams through the ring, whose slots and
    # mbarrier phases carry over from layer to layer; ragged F (a short last
    # piece), INT4, gated and plain fp16 rows
    ("int4-ring", small(CONFIGS["c5"], d=1280, F=16390, rank=1024), 3),
    ("gated-ring", small(CONFIGS["c4"], d=1024, F=16390, rank=1024), 3),
    ("fp16-ring", small(CONFIGS["c2"], d=1024, F=16390, rank=1024), 3),
])
def test_stack_p2_ring_matches_oracle(name, cfg, L):
    _check_stack(cfg, L, p2_ring=True)


def test_stack_rank_beyond_the_ring_runs_per_step_kernels():
    """Rank 4096: a 16-row P2 unit is 128 KB, so fewer than two ring slots fit
    in shared memory; the plan drops the persistent kernel and the step runs on
    the per-step kernels, still matching the oracle layer by layer."""
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    cfg = small(CONFIGS["c2"], d=4096, F=5000, rank=4096)
    ws = [make_layer(cfg, l, device=DEV) for l in range(2)]
    st = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    assert P.pi_stack_plan(st.desc, 2, st.ranks).fused == 0
    assert P.pi_launches_per_layer(st.desc) > 1
    del st, ws
    _check_stack(cfg, 2)


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


def test_grid_barrier_wait_runs_out_and_next_step_matches_oracle():
    """The persistent kernel's own grid barrier runs out.  The workspace's
    barrier epoch is pushed far ahead of the arrival counter (a host-side
    change of the caller-owned workspace), so the first barrier's target is
    never reached; with a 5 ms wait limit every block gives up, the device
    status reads PI_ERR_TIMEOUT and the context stays usable.  After the
    workspace is zero-filled again the next step matches the oracle."""
    import time
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    ws = [make_layer(cfg, l, device=DEV) for l in range(2)]
    st = DecodeStack(ws, batch=1, tau=cfg.tau, eps=cfg.rms_eps)
    x = make_tokens(cfg, 0, 1, device=DEV)
    y0 = st.step(x).clone()
    torch.cuda.synchronize()
    assert P.pi_last_device_status() == 0
    epoch = st.workspace[0:8].view(torch.int64)
    epoch += 1000                               # 1000 barriers that never happened
    P.pi_debug_set_wait_timeout(5_000_000)
    try:
        t0 = time.perf_counter()
        st.step(x)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        P.pi_debug_set_wait_timeout(0)
    assert P.pi_last_device_status() == 4       # PI_ERR_TIMEOUT, then cleared
    assert P.pi_last_device_status() == 0
    assert elapsed < 1.0, f"the barrier gave up after {elapsed:.3f} s, not after its 5 ms limit"
    st.workspace.zero_()
    xs, y1 = st.step_trace(x)
    torch.cuda.synchronize()
    assert P.pi_last_device_status() == 0
    assert torch.equal(y1, y0)
    host = oracle.host_layer(ws[1].to("cpu"))
    close(y1[0].cpu().numpy(), oracle.ffn_masked(xs[1][0].cpu(), host, _mask_of(P, st)), "step after timeout")


def test_tensor_core_stage_wait_runs_out_and_frees_tensor_memory():
    """A tcgen05 row kernel (batched FC1, 16 tokens) whose stage waits run out:
    with a 1 ns wait limit the first wait that is not already satisfied gives
    up, the block drains its own copies and MMAs, frees its tensor memory and
    returns, and the status reads PI_ERR_TIMEOUT.  The same call afterwards
    (which allocates tensor memory on every SM again) gives the bits of a
    clean run."""
    P = _pi()
    cfg = small(CONFIGS["c3"], d=1024, F=4096, rank=64)
    B = 16
    w = make_layer(cfg, 0, device=DEV)
    x = make_tokens(cfg, 0, B, device=DEV)
    desc = P.layer_desc(w, B)
    wsb = torch.zeros(P.pi_workspace_bytes(desc), dtype=torch.uint8, device=DEV)
    mask = torch.zeros(B, (w.F + 31) // 32, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, wsb)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    wsx = P.weights_struct(w)
    h_ref = torch.zeros(w.F * B, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask, h_ref, wsb)
    torch.cuda.synchronize()
    assert P.pi_last_device_status() == 0
    h_bad = torch.zeros_like(h_ref)
    P.pi_debug_set_wait_timeout(1)
    try:
        P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask, h_bad, wsb)
        torch.cuda.synchronize()
    finally:
        P.pi_debug_set_wait_timeout(0)
    assert P.pi_last_device_status() == 4
    for _ in range(3):
        h = torch.zeros_like(h_ref)
        P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask, h, wsb)
        torch.cuda.synchronize()
        assert P.pi_last_device_status() == 0
        assert torch.equal(h, h_ref)
