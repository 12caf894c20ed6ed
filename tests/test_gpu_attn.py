"""Parity of the head-sparse attention block (pi_attn_heads) with the oracle.

Per sequence of the batch: the head mask against the oracle's head predictor
(identical outside its guard band), y against oracle.attn_heads run with the
GPU's own mask (max-abs 2e-3, rel-L2 1e-3), the token's key and value in the
cache equal to the binary16 rounding of a value within the fp32 evaluation
bound of the exact projection (almost all of them the oracle's own rounding),
and every other cache position unchanged bit for bit.  Shapes: small blocks with ragged cache
lengths (the first and the last position included), multi-head and grouped
KV heads, head_dim 64 and 128, batches that take each output-projection path,
and the full OPT-6.7B, LLaMA-70B and OPT-175B block shapes at batch 1.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import close, half_matches, mask_matches, unpack_mask
from synth import ATTN_CONFIGS, make_attn, make_kv_cache, small_attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def P():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    return P


def _tokens(d, B, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, d, generator=g).to(torch.float16)


def _run(P, cfg, w, x, lengths, kc, vc, tau):
    B = x.shape[0]
    dev = "cuda"
    wd = w.to(dev)
    desc = P.attn_desc(wd, B, kc.shape[2])
    ws = torch.empty(P.pi_attn_workspace_bytes(desc), dtype=torch.uint8, device=dev)
    assert ws.numel() > 0
    kd, vd = kc.to(dev).contiguous(), vc.to(dev).contiguous()
    pos = torch.tensor(lengths, dtype=torch.int32, device=dev)
    mask = torch.zeros(B, (w.H + 31) // 32, dtype=torch.int32, device=dev)
    y = torch.zeros(B, w.d, dtype=torch.float32, device=dev)
    st = P.attn_weights_struct(wd)
    xd = x.to(dev)
    P.pi_attn_heads(desc, xd, st, kd, vd, pos, tau, mask, y, ws)
    torch.cuda.synchronize()
    assert P.pi_last_device_status() == 0

    def again():
        # the struct holds raw pointers: wd and xd must outlive every call
        P.pi_attn_heads(desc, xd, P.attn_weights_struct(wd), kd, vd, pos, tau, mask, y, ws)
        return y

    return dict(y=y.cpu().numpy(), mask=mask.cpu().numpy().view(np.uint32), kc=kd.cpu(), vc=vd.cpu(), run=again)


def _check(cfg, w, x, lengths, kc, vc, g, what):
    B = x.shape[0]
    H, KVH, dh = w.H, w.KVH, w.dh
    for b in range(B):
        pr = oracle.attn_predict(x[b], w.p1, w.p2, w.bp, cfg.tau)
        mask_matches(g["mask"][b], pr, H, cfg.tau, f"{what} head mask b={b}")
    ref = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, g["mask"], kc, vc, lengths, H, KVH, dh)
    for b in range(B):
        close(g["y"][b], ref["y"][b], f"{what} y b={b}")
    kg = g["kc"].numpy().view(np.uint16)
    vg = g["vc"].numpy().view(np.uint16)
    nkv = KVH * dh
    for b, p in enumerate(lengths):
        # untouched positions: bit for bit
        keep = np.ones(kg.shape[2], bool)
        keep[p] = False
        np.testing.assert_array_equal(kg[b][:, keep], kc.numpy().view(np.uint16)[b][:, keep])
        np.testing.assert_array_equal(vg[b][:, keep], vc.numpy().view(np.uint16)[b][:, keep])
        # the token's key and value: the binary16 rounding of a value within
        # the fp32 evaluation bound of the exact projection
        pre, band = ref["kv_pre"][b], ref["kv_band"][b]
        half_matches(kg[b, :, p].ravel(), pre[:nkv], band[:nkv], f"{what} key b={b}")
        half_matches(vg[b, :, p].ravel(), pre[nkv:], band[nkv:], f"{what} value b={b}")
        exact = (kg[b, :, p].ravel() == ref["kcache"][b, :, p].ravel()).mean()
        assert exact > 0.95, f"{what} key b={b}: only {exact:.3f} of the elements equal the oracle's rounding"
    return ref


CASES = [
    # (H, KVH, dh, d, smax, lengths)
    (8, 8, 64, 256, 64, [0, 5, 63]),
    (16, 4, 128, 512, 80, [17]),
    (12, 3, 64, 384, 40, [39, 0, 20, 7, 33]),
    (24, 24, 128, 1024, 96, [1, 50, 95]),
]


@pytest.mark.parametrize("H,KVH,dh,d,smax,lengths", CASES)
def test_attn_heads_small(P, H, KVH, dh, d, smax, lengths):
    cfg = small_attn(ATTN_CONFIGS["c4"], d=d, heads=H, kv_heads=KVH, head_dim=dh, rank=8, max_seq=smax,
                     index=60 + H + dh)
    w = make_attn(cfg)
    kc, vc = make_kv_cache(cfg, lengths, seed=3)
    x = _tokens(d, len(lengths), 11 + H)
    g = _run(P, cfg, w, x, lengths, kc, vc, cfg.tau)
    _check(cfg, w, x, lengths, kc, vc, g, f"H{H}/KVH{KVH}/dh{dh}")
    on = unpack_mask(g["mask"].ravel(), H * len(lengths))
    assert 0 < on.sum() < on.size, "the synthetic head predictor should keep some heads and drop others"


@pytest.mark.parametrize("B,d", [(2, 512), (5, 512), (8, 512), (11, 512), (16, 512), (32, 512), (16, 320)])
def test_attn_heads_batches(P, B, d):
    """Batches that take each projection and output-projection path: per-token
    (1..4, 9..15, and widths off the tensor-core tiles), streamed (5..8),
    tensor cores (16..32)."""
    cfg = small_attn(ATTN_CONFIGS["c2"], d=d, heads=8, kv_heads=8, head_dim=64, rank=8, max_seq=48,
                     index=90 + B)
    w = make_attn(cfg)
    lengths = [(7 * b + 3) % 48 for b in range(B)]
    kc, vc = make_kv_cache(cfg, lengths, seed=B)
    x = _tokens(cfg.d, B, 200 + B)
    g = _run(P, cfg, w, x, lengths, kc, vc, cfg.tau)
    _check(cfg, w, x, lengths, kc, vc, g, f"B{B} d{d}")


def test_attn_heads_no_head_and_all_heads(P):
    cfg = small_attn(ATTN_CONFIGS["c2"], d=256, heads=8, kv_heads=2, head_dim=64, rank=8, max_seq=32, index=77)
    w = make_attn(cfg)
    lengths = [9, 30]
    kc, vc = make_kv_cache(cfg, lengths, seed=8)
    x = _tokens(cfg.d, 2, 5)
    for tau, expect in ((1e4, 0), (-1e4, 8)):
        g = _run(P, cfg, w, x, lengths, kc, vc, tau)
        on = unpack_mask(g["mask"].ravel(), 64)
        for b in range(2):
            assert int(on[b * 32:(b * 32) + 8].sum()) == expect
        ref = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, g["mask"], kc, vc, lengths, 8, 2, 64)
        for b in range(2):
            close(g["y"][b], ref["y"][b], f"tau={tau} b={b}")
        if expect == 0:
            np.testing.assert_allclose(g["y"], np.broadcast_to(w.bo.double().numpy(), g["y"].shape), rtol=0,
                                       atol=0)


def test_attn_heads_repeatable_bitwise(P):
    cfg = small_attn(ATTN_CONFIGS["c3"], d=512, heads=16, kv_heads=16, head_dim=128, rank=8, max_seq=128,
                     index=81)
    w = make_attn(cfg)
    lengths = [100, 3, 64]
    kc, vc = make_kv_cache(cfg, lengths, seed=9)
    x = _tokens(cfg.d, 3, 6)
    g = _run(P, cfg, w, x, lengths, kc, vc, cfg.tau)
    y1 = g["y"].copy()
    y = g["run"]()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y.cpu().numpy(), y1)


def test_attn_heads_bad_position_sets_status(P):
    cfg = small_attn(ATTN_CONFIGS["c2"], d=256, heads=8, kv_heads=8, head_dim=64, rank=8, max_seq=16, index=83)
    w = make_attn(cfg).to("cuda")
    desc = P.attn_desc(w, 2, 16)
    ws = torch.empty(P.pi_attn_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    kc, vc = make_kv_cache(cfg, [4, 4], seed=1)
    kd, vd = kc.cuda(), vc.cuda()
    pos = torch.tensor([4, 16], dtype=torch.int32, device="cuda")
    mask = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
    y = torch.zeros(2, 256, device="cuda")
    P.pi_attn_heads(desc, _tokens(256, 2, 1).cuda(), P.attn_weights_struct(w), kd, vd, pos, -1e4, mask, y, ws)
    assert P.pi_last_device_status() == P.binding.PI_ERR_INVALID_ARG
    assert P.pi_last_device_status() == 0
    np.testing.assert_array_equal(kd[1].cpu().numpy(), kc[1].numpy())
    np.testing.assert_allclose(y[1].cpu().double().numpy(), w.bo.cpu().double().numpy(), rtol=0, atol=0)
    assert (kd[0, :, 4] != 0).any()


@pytest.mark.parametrize("key", ["c2", "c4", "c5"])
def test_attn_heads_full_shape(P, key):
    """The full block shapes at batch 1 with a decode-length cache."""
    cfg = ATTN_CONFIGS[key]
    w = make_attn(cfg, 0, device="cuda").to("cpu")
    lengths = [cfg.prompt + 77]
    kc, vc = make_kv_cache(cfg, lengths, seed=1, max_seq=512)
    x = _tokens(cfg.d, 1, 3)
    g = _run(P, cfg, w, x, lengths, kc, vc, cfg.tau)
    _check(cfg, w, x, lengths, kc, vc, g, key)
