"""Parity of the INT4 batched path (streamed CUDA-core kernels, batch 2..16,
ReLU FFN) against the fp64 CPU oracle, through the C ABI.

FC1 works on 256-element K-chunks of the packed rows (codes + group scales),
FC2 on 256-column tiles; both split (tile x chunk) work evenly over the CTAs
and add the per-CTA partials in a fixed order.  The cases cover ragged row
tiles, several tiles per CTA, FC2 run in two token passes (batch > 8), rows
that FC1 found dead (FC2 zero-fills them), tiny and empty unions.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close, mask_matches
from tests.test_gpu_tc import _check_fc, _masks, _pi, _ws

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = [
    ("int4-d512", small(CONFIGS["c5"], d=512, F=3000, rank=64)),
    ("int4-d1024", small(CONFIGS["c5"], d=1024, F=4099, rank=64)),
]


@pytest.mark.parametrize("kind,cfg", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("batch", [2, 3, 4, 5, 8, 9, 12, 16])
def test_st4_fc1_fc2_parity(kind, cfg, batch):
    P = _pi()
    w = make_layer(cfg, 0, device=DEV)
    wh = w.to("cpu")
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    mask, idx, cnt = _masks(P, w, cfg, x, desc, ws, batch)
    _check_fc(P, w, wh, x, desc, ws, mask, idx, cnt, batch, f"{kind} B={batch}")


@pytest.mark.parametrize("batch", [4, 16])
def test_st4_many_tiles_per_cta(batch):
    """More 128-row FC1 tiles than CTAs, FC2 ranges crossing column tiles."""
    P = _pi()
    cfg = small(CONFIGS["c5"], d=256, F=72000, rank=32, mean_rate=0.35)
    w = make_layer(cfg, 0, device=DEV)
    wh = w.to("cpu")
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    mask, idx, cnt = _masks(P, w, cfg, x, desc, ws, batch)
    n = int(cnt.item())
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert n > 128 * sms, n
    _check_fc(P, w, wh, x, desc, ws, mask, idx, cnt, batch, "int4 many tiles",
              sample=sorted({0, batch // 2, batch - 1}))


@pytest.mark.parametrize("batch", [4, 16])
def test_st4_tiny_and_empty_union(batch):
    P = _pi()
    cfg = CASES[0][1]
    w = make_layer(cfg, 0, device=DEV)
    wh = w.to("cpu")
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    W = (w.F + 31) // 32
    words = np.zeros((batch, W), np.uint32)
    rng = np.random.default_rng(7)
    for r in rng.choice(w.F, size=5, replace=False):
        words[rng.integers(batch), r // 32] |= np.uint32(1 << (r % 32))
    mask = torch.from_numpy(words.view(np.int32)).to(DEV)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    torch.cuda.synchronize()
    assert int(cnt.item()) == 5
    _check_fc(P, w, wh, x, desc, ws, mask, idx, cnt, batch, "int4 tiny union")
    # empty list: y = b2 for every token
    cnt.zero_()
    h = torch.zeros(w.F * batch, dtype=torch.float32, device=DEV)
    y = torch.full((batch, w.d), float("nan"), dtype=torch.float32, device=DEV)
    wsx = P.weights_struct(w)
    P.pi_sparse_fc1(desc, x, wsx, idx, cnt, None, h, ws)
    P.pi_sparse_fc2(desc, h, idx, cnt, wsx, y, ws)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), np.broadcast_to(w.b2.float().cpu().numpy(), (batch, w.d)))


@pytest.mark.parametrize("batch", [6, 16])
def test_st4_layer_matches_oracle(batch):
    """Whole layer (FC2 skips the rows FC1 found dead for every token): each
    row equals the oracle's masked FFN of its token's own mask."""
    P = _pi()
    cfg = CASES[1][1]
    w = make_layer(cfg, 0, device=DEV)
    wh = oracle.host_layer(w.to("cpu"))
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = _ws(P, desc)
    y = torch.empty(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_ffn_layer(desc, x, P.weights_struct(w), cfg.tau, ws, y)
    torch.cuda.synchronize()
    lay = P.pi_workspace_layout(desc)
    W = (w.F + 31) // 32
    mask = ws[lay.mask:lay.mask + 4 * batch * W].view(torch.int32).cpu().numpy().view(np.uint32).reshape(batch, W)
    yb = y.cpu().numpy()
    for b in range(batch):
        mask_matches(mask[b], oracle.predict(x[b].cpu(), wh, cfg.tau), w.F, cfg.tau, f"int4 token {b}")
        close(yb[b], oracle.ffn_masked(x[b].cpu(), wh, mask[b]), f"int4 layer token {b}")
    # bitwise repeatable
    y2 = torch.empty_like(y)
    P.pi_ffn_layer(desc, x, P.weights_struct(w), cfg.tau, ws, y2)
    torch.cuda.synchronize()
    assert np.array_equal(yb, y2.cpu().numpy())
    assert P.pi_last_device_status() == 0
