"""Second tier of FC rows (the pages' hot/cold neuron placement, with the
cold neurons' rows in the host's memory): storage rows past the hot prefix are
read from separate arrays, here pinned host memory the GPU reads directly (on
a Grace-Blackwell system, Grace memory over NVLink-C2C) or a separate device
buffer.  The results must be the bits of the single-tier per-token path (same
kernels, same order) and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _split(w, n_hot, where):
    """The rows of w from n_hot on, copied to `where` ("host": pinned host
    memory, "device": a separate device buffer)."""
    def cold(t):
        if t is None:
            return None
        c = t[n_hot:].contiguous()
        return c.cpu().pin_memory() if where == "host" else c.clone()
    if w.int4:
        return dict(w1=cold(w.w1_q), w1_scales=cold(w.w1_s), w2t=cold(w.w2t_q), w2t_scales=cold(w.w2t_s))
    return dict(w1=cold(w.w1), wu=cold(w.wu), w2t=cold(w.w2t))


@pytest.mark.parametrize("kind,cfg,batch,where", [
    ("fp16", small(CONFIGS["c2"], d=1024, F=4096, rank=64), 1, "host"),
    ("fp16", small(CONFIGS["c2"], d=1024, F=4096, rank=64), 1, "device"),
    ("gated", small(CONFIGS["c4"], d=1024, F=3000, rank=64), 1, "host"),
    ("int4", small(CONFIGS["c5"], d=1024, F=4100, rank=64), 1, "host"),
    ("int4-b3", small(CONFIGS["c5"], d=1024, F=4100, rank=64), 3, "host"),
    ("fp16-b5", small(CONFIGS["c3"], d=1024, F=4096, rank=64), 5, "host"),
])
def test_tiered_fc_matches_single_tier_and_oracle(kind, cfg, batch, where):
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    w = make_layer(cfg, 0, device=DEV)
    # a short first tier, so that the predicted rows (mostly from the hot
    # prefix of the table) fall on both sides of the split
    n_hot = 96
    tensors = _split(w, n_hot, where)
    cold = P.cold_tier(n_hot, **tensors)
    x = make_tokens(cfg, 0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = torch.zeros(P.pi_workspace_bytes(desc), dtype=torch.uint8, device=DEV)
    mask = torch.zeros(batch, (w.F + 31) // 32, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    wsx = P.weights_struct(w)
    m = mask if batch > 1 else None
    h_t = torch.zeros(w.F * batch, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc1_tiered(desc, x, wsx, cold, idx, cnt, m, h_t)
    y_t = torch.zeros(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc2_tiered(desc, h_t, idx, cnt, wsx, cold, y_t, ws)
    # every row in the first tier: the same kernels and order
    all_hot = P.cold_tier(w.F)
    h_1 = torch.zeros_like(h_t)
    P.pi_sparse_fc1_tiered(desc, x, wsx, all_hot, idx, cnt, m, h_1)
    y_1 = torch.zeros_like(y_t)
    P.pi_sparse_fc2_tiered(desc, h_1, idx, cnt, wsx, all_hot, y_1, ws)
    torch.cuda.synchronize()
    c = int(cnt.item())
    assert c > 0 and (idx[:c] >= n_hot).any() and (idx[:c] < n_hot).any(), "rows of both tiers listed"
    assert torch.equal(h_t, h_1) and torch.equal(y_t, y_1), f"{kind}/{where}: tiers change the bits"
    if batch == 1:
        # batch 1 single-tier entry points take the same per-token kernels
        h_s = torch.zeros_like(h_t)
        P.pi_sparse_fc1(desc, x, wsx, idx, cnt, None, h_s, ws)
        torch.cuda.synchronize()
        assert torch.equal(h_t, h_s)
    host = oracle.host_layer(w.to("cpu"))
    ix = idx[:c].cpu().numpy()
    for b in range(batch):
        bits = mask[b].cpu().numpy().view(np.uint32)
        close(y_t[b].cpu().numpy(), oracle.ffn_masked(x[b].cpu(), host, bits), f"{kind}/{where} token {b}")


def test_tiered_layer_matches_oracle_and_rejects_bad_tiers():
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=64)
    w = make_layer(cfg, 0, device=DEV)
    n_hot = 96
    keep = _split(w, n_hot, "host")
    cold = P.cold_tier(n_hot, **keep)
    x = make_tokens(cfg, 3, 1, device=DEV)
    desc = P.layer_desc(w, 1)
    ws = torch.zeros(P.pi_workspace_bytes(desc), dtype=torch.uint8, device=DEV)
    y = torch.zeros(1, w.d, dtype=torch.float32, device=DEV)
    P.pi_ffn_layer_tiered(desc, x, P.weights_struct(w), cold, cfg.tau, ws, y)
    torch.cuda.synchronize()
    lay = P.pi_workspace_layout(desc)
    W = (w.F + 31) // 32
    mask = ws[lay.mask:lay.mask + 4 * W].view(torch.int32).cpu().numpy().view(np.uint32)
    close(y[0].cpu().numpy(), oracle.ffn_masked(x[0].cpu(), oracle.host_layer(w.to("cpu")), mask), "tiered layer")
    for bad in (P.cold_tier(-1), P.cold_tier(w.F + 1), P.cold_tier(n_hot)):   # the last: no cold arrays
        with pytest.raises(P.PiError) as e:
            P.pi_ffn_layer_tiered(desc, x, P.weights_struct(w), bad, cfg.tau, ws, y)
        assert e.value.status == 1
