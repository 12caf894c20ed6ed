"""Parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Each kernel is checked in isolation on the same seeded inputs: the predictor
mask (bit-exact outside the guard band), the compaction (bit-exact, given the
GPU's mask), FC1 and FC2 (given the same index list / FC1 outputs), the
whole layer and the inter-layer normalisation.  Shapes run from tiny ragged
cases up to the full workload shapes.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close, half_matches, mask_matches, unpack_mask

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _pi():
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    return P


def _layer(cfg, l=0):
    w = make_layer(cfg, l, device=DEV)
    return w, w.to("cpu")


def _ws(P, desc):
    return torch.zeros(P.pi_workspace_bytes(desc), dtype=torch.uint8, device=DEV)


def _run_layer(P, w, x, tau, batch=1):
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    y = torch.empty(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_ffn_layer(desc, x, P.weights_struct(w), tau, ws, y)
    lay = P.pi_workspace_layout(desc)
    torch.cuda.synchronize()
    W = (w.F + 31) // 32
    mask = ws[lay.mask:lay.mask + 4 * batch * W].view(torch.int32).cpu().numpy().view(np.uint32).reshape(batch, W)
    n = int(ws[lay.count:lay.count + 4].view(torch.int32).item())
    idx = ws[lay.idx:lay.idx + 4 * n].view(torch.int32).cpu().numpy() if n else np.zeros(0, np.int32)
    h = ws[lay.h:lay.h + 4 * w.F * batch].view(torch.float32).cpu().numpy()
    return y.cpu().numpy(), mask, idx, n, h


SMALL = [
    dict(d=256, F=1000, rank=32),          # F not a multiple of 32 (ragged last word)
    dict(d=136, F=64, rank=8),             # d not a multiple of 32, tiny F
    dict(d=1024, F=4099, rank=64),
]


@pytest.mark.parametrize("shape", SMALL)
def test_predict_mask_parity_small(shape):
    P = _pi()
    cfg = small(CONFIGS["c1"], **shape)
    w, wh = _layer(cfg)
    xs = make_tokens(cfg, 0, 4, device=DEV)
    for t in range(4):
        desc = P.layer_desc(w, 1)
        ws = _ws(P, desc)
        mask = torch.zeros((w.F + 31) // 32, dtype=torch.int32, device=DEV)
        P.pi_predict(desc, xs[t:t + 1], w.p1, w.p2, w.b1, cfg.tau, mask, ws)
        torch.cuda.synchronize()
        o = oracle.predict(xs[t].cpu(), wh, cfg.tau)
        mask_matches(mask.cpu().numpy().view(np.uint32), o, w.F, cfg.tau, f"token {t}")


@pytest.mark.parametrize("batch", [2, 3, 4, 8, 11])
def test_predict_batched_matches_per_token(batch):
    P = _pi()
    cfg = small(CONFIGS["c3"], d=512, F=2080, rank=96, per_layer_rates=())
    w, wh = _layer(cfg)
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    W = (w.F + 31) // 32
    mask = torch.zeros(batch, W, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)
    torch.cuda.synchronize()
    m = mask.cpu().numpy().view(np.uint32)
    for b in range(batch):
        mask_matches(m[b], oracle.predict(x[b].cpu(), wh, cfg.tau), w.F, cfg.tau, f"token {b}")


@pytest.mark.parametrize("F,density", [(1, 1.0), (31, 0.5), (32, 1.0), (33, 0.3), (1000, 0.05),
                                       (49152, 0.06), (49152, 0.0), (65536 + 7, 0.9)])
def test_compact_bit_exact(F, density):
    P = _pi()
    rng = np.random.default_rng(F)
    W = (F + 31) // 32
    bits = rng.random(W * 32) < density
    bits[F:] = False
    words = np.packbits(bits.reshape(-1, 32)[:, ::-1], axis=1).view(">u4").ravel().astype(np.uint32)
    table = rng.permutation(F).astype(np.int32)
    desc = P.desc_of(8, F, 8, 1)
    m = torch.from_numpy(words.view(np.int32)).to(DEV)
    tb = torch.from_numpy(table).to(DEV)
    idx = torch.full((F,), -7, dtype=torch.int32, device=DEV)
    orig = torch.full((F,), -7, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, m, tb, idx, orig, cnt)
    torch.cuda.synchronize()
    oi, oo, on = oracle.compact(words, F, table)
    n = int(cnt.item())
    assert n == on
    assert np.array_equal(idx.cpu().numpy()[:n], oi)
    assert np.array_equal(orig.cpu().numpy()[:n], oo)


def test_compact_union_of_batch():
    P = _pi()
    rng = np.random.default_rng(3)
    B, F = 5, 3000
    W = (F + 31) // 32
    bits = rng.random((B, W * 32)) < 0.04
    bits[:, F:] = False
    words = np.packbits(bits.reshape(B, W, 32)[:, :, ::-1], axis=2).view(">u4").reshape(B, W).astype(np.uint32)
    desc = P.desc_of(8, F, 8, B)
    idx = torch.zeros(F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, torch.from_numpy(words.view(np.int32)).to(DEV), None, idx, None, cnt)
    torch.cuda.synchronize()
    oi, _, on = oracle.compact(oracle.mask_union(words, F), F)
    assert int(cnt.item()) == on and np.array_equal(idx.cpu().numpy()[:on], oi)


def _fc_case(P, cfg, batch, layer=0):
    w, wh = _layer(cfg, layer)
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    W = (w.F + 31) // 32
    mask = torch.zeros(batch, W, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    torch.cuda.synchronize()
    return w, wh, x, desc, ws, mask, idx, cnt


FC_CASES = [
    ("fp16", small(CONFIGS["c1"], d=256, F=1000, rank=32)),
    ("gated", small(CONFIGS["c4"], d=512, F=1500, rank=64)),
    ("int4", small(CONFIGS["c5"], d=512, F=2000, rank=64)),
]


@pytest.mark.parametrize("kind,cfg", FC_CASES, ids=[c[0] for c in FC_CASES])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_fc1_fc2_parity(kind, cfg, batch):
    P = _pi()
    w, wh, x, desc, ws, mask, idx, cnt = _fc_case(P, cfg, batch)
    n = int(cnt.item())
    assert n > 0
    h = torch.full((w.F * batch,), float("nan"), dtype=torch.float32, device=DEV)
    wsx = P.weights_struct(w)
    P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask if batch > 1 else None, h, ws)
    y = torch.empty(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc2(desc, h, idx, cnt, wsx, y, ws)
    torch.cuda.synchronize()
    idx_h = idx.cpu().numpy()[:n]
    hg = h.cpu().numpy()[: n * batch].reshape(n, batch)
    mk = mask.cpu().numpy().view(np.uint32)
    for b in range(batch):
        ho = oracle.fc1(x[b].cpu(), wh, idx_h)
        if batch > 1:
            own = unpack_mask(mk[b], w.F)[idx_h]
            ho = np.where(own, ho, 0.0)
        close(hg[:, b], ho, f"{kind} fc1 token {b}")
        yo = oracle.fc2(hg[:, b].astype(np.float64), wh, idx_h)
        close(y[b].cpu().numpy(), yo, f"{kind} fc2 token {b}")


@pytest.mark.parametrize("kind,cfg", FC_CASES, ids=[c[0] for c in FC_CASES])
@pytest.mark.parametrize("batch", [1, 4])
def test_layer_parity_small(kind, cfg, batch):
    P = _pi()
    w, wh = _layer(cfg)
    x = make_tokens(cfg, 0, batch, device=DEV)
    y, mask, idx, n, _ = _run_layer(P, w, x, cfg.tau, batch)
    for b in range(batch):
        o = oracle.predict(x[b].cpu(), wh, cfg.tau)
        mask_matches(mask[b], o, w.F, cfg.tau, f"{kind} token {b}")
        close(y[b], oracle.ffn_masked(x[b].cpu(), wh, mask[b]), f"{kind} layer token {b}")
    oi, _, on = oracle.compact(oracle.mask_union(mask, w.F), w.F)
    assert n == on and np.array_equal(idx, oi)


def test_layer_empty_and_full_masks():
    P = _pi()
    cfg = small(CONFIGS["c1"], d=256, F=1000, rank=32)
    w, wh = _layer(cfg)
    x = make_tokens(cfg, 0, 1, device=DEV)
    # tau above every score: nothing active, y == b2 exactly
    y, mask, idx, n, _ = _run_layer(P, w, x, 1e30)
    assert n == 0 and not mask.any()
    assert np.array_equal(y[0], wh.b2.float().numpy())
    # tau below every score: every neuron active, y == dense FFN
    y, mask, idx, n, _ = _run_layer(P, w, x, -1e30)
    assert n == w.F
    close(y[0], oracle.ffn_dense(x[0].cpu(), wh), "all-active layer")


def test_rmsnorm_parity():
    P = _pi()
    rng = np.random.default_rng(5)
    for d, B in ((768, 1), (4096, 3), (12288, 2), (8, 1), (20000, 2)):
        y = (rng.standard_normal((B, d)) * rng.uniform(0.01, 3.0)).astype(np.float32)
        yd = torch.from_numpy(y).to(DEV)
        x = torch.empty(B, d, dtype=torch.float16, device=DEV)
        P.pi_rmsnorm_half(d, B, yd, 1e-6, x)
        torch.cuda.synchronize()
        xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
        for b in range(B):
            _, pre, band = oracle.rmsnorm_half(y[b].astype(np.float64), 1e-6)
            half_matches(xb[b], pre, band, f"rmsnorm d={d}")


def test_layer_repeatable_bitwise():
    P = _pi()
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    w, _ = _layer(cfg)
    x = make_tokens(cfg, 0, 1, device=DEV)
    y1 = _run_layer(P, w, x, cfg.tau)[0]
    y2 = _run_layer(P, w, x, cfg.tau)[0]
    assert np.array_equal(y1, y2)


def test_invalid_arguments_rejected():
    P = _pi()
    cfg = small(CONFIGS["c1"], d=256, F=1000, rank=32)
    w, _ = _layer(cfg)
    x = make_tokens(cfg, 0, 1, device=DEV)
    desc = P.layer_desc(w, 1)
    y = torch.empty(1, w.d, dtype=torch.float32, device=DEV)
    small_ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(P.PiError) as e:
        P.pi_ffn_layer(desc, x, P.weights_struct(w), cfg.tau, small_ws, y)
    assert e.value.status == 5
    bad = P.desc_of(250, w.F, w.r, 1)                   # d not a multiple of 8
    with pytest.raises(P.PiError) as e:
        P.pi_ffn_layer(bad, x, P.weights_struct(w), cfg.tau, _ws(P, desc), y)
    assert e.value.status == 1
