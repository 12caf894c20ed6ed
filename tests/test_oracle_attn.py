"""Pins of the oracle's head-sparse attention block (oracle_attn_heads).

- a step worked by hand, for every head mask (tests/golden/attn_small.txt);
- one cached position (pos = 0): softmax over a single position is 1, so the
  block reduces to the value projection times the output projection;
- every head active: equals dense multi-head attention with
  torch.nn.functional.scaled_dot_product_attention (fp64) as the attention;
- grouped key/value heads equal multi-head attention with each KV head's rows
  and cache repeated for its group;
- no head active: y = bo exactly, the cache still receives the token;
- the head predictor's mask is the strict threshold of the scores computed
  from the predictor's own factors.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from synth import ATTN_CONFIGS, make_attn, make_kv_cache, small_attn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out.setdefault(k, []).append([float(t) for t in v])
    return out


def _h(a):
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def _f(t):
    """fp16 torch tensor or bits -> float64 numpy."""
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().double().numpy()
    return np.asarray(t).view(np.float16).astype(np.float64)


def test_golden_hand_worked_step():
    g = _fixture("attn_small.txt")
    d, H, KVH, dh, pos = (int(g[k][0][0]) for k in ("d", "H", "KVH", "dh", "pos"))
    x = _h(g["x"][0])[None]
    wqkv = _h(g["wqkv"])
    bqkv = _h(g["bqkv"][0])
    wot = _h(g["wot"])
    bo = _h(g["bo"][0])
    smax = 4
    kc = np.zeros((1, KVH, smax, dh), np.float16)
    vc = np.zeros((1, KVH, smax, dh), np.float16)
    kc[0, 0, 0] = g["k0"][0]
    vc[0, 0, 0] = g["v0"][0]
    for m in (3, 1, 2, 0):
        r = oracle.attn_heads(x, wqkv, bqkv, wot, bo, np.array([[m]], np.uint32), kc, vc, [pos], H, KVH, dh)
        np.testing.assert_allclose(r["y"][0], g[f"y_mask{m}"][0], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(_f(r["kcache"])[0, 0, pos], g["k_new"][0])
        np.testing.assert_array_equal(_f(r["vcache"])[0, 0, pos], g["v_new"][0])
        # the earlier position is untouched
        np.testing.assert_array_equal(_f(r["vcache"])[0, 0, 0], g["v0"][0])
        if m & 1:
            np.testing.assert_allclose(r["o"][0, :dh], g["o0"][0], rtol=0, atol=1e-12)
        else:
            assert not r["o"][0, :dh].any()
        if m & 2:
            np.testing.assert_allclose(r["o"][0, dh:], g["o1"][0], rtol=0, atol=1e-12)


def _block(H=6, KVH=3, dh=16, d=64, smax=24, seed=0):
    cfg = small_attn(ATTN_CONFIGS["c4"], d=d, heads=H, kv_heads=KVH, head_dim=dh, rank=min(8, H) // 8 * 8 or 8,
                     max_seq=smax, index=40 + seed)
    w = make_attn(cfg)
    return cfg, w


def _x(d, B, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, d, generator=g).to(torch.float16)


def _mask_all(H, B):
    words = (H + 31) // 32
    m = np.zeros((B, words), np.uint32)
    for h in range(H):
        m[:, h // 32] |= np.uint32(1 << (h % 32))
    return m


def _dense_reference(x, w, kc, vc, pos, heads):
    """Dense attention over the given heads: numpy projections, torch SDPA in
    fp64 as the attention, the new key/value rounded to binary16 first."""
    H, KVH, dh = w.H, w.KVH, w.dh
    G = H // KVH
    W = _f(w.wqkv)
    bq = _f(w.bqkv)
    Wo = _f(w.wot)
    bo = _f(w.bo)
    xv = _f(x)
    proj = W @ xv + bq
    kn = proj[H * dh:(H + KVH) * dh].reshape(KVH, dh).astype(np.float16).astype(np.float64)
    vn = proj[(H + KVH) * dh:].reshape(KVH, dh).astype(np.float16).astype(np.float64)
    K = _f(kc).copy()
    V = _f(vc).copy()
    K[:, pos] = kn
    V[:, pos] = vn
    y = bo.copy()
    for h in heads:
        g = h // G
        q = torch.from_numpy(proj[h * dh:(h + 1) * dh])[None, None, None]
        k = torch.from_numpy(K[g, :pos + 1])[None, None]
        v = torch.from_numpy(V[g, :pos + 1])[None, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v).numpy().reshape(dh)
        y += Wo[h * dh:(h + 1) * dh].T @ o
    return y


@pytest.mark.parametrize("H,KVH", [(6, 6), (6, 2), (4, 1)])
def test_all_heads_equal_dense_attention_with_sdpa(H, KVH):
    cfg, w = _block(H=H, KVH=KVH, seed=H + KVH)
    lengths = [0, 5, 17]
    kc, vc = make_kv_cache(cfg, lengths, seed=1)
    x = _x(cfg.d, len(lengths), 3)
    r = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, _mask_all(H, len(lengths)), kc, vc, lengths, H, KVH,
                          cfg.head_dim)
    for b, pos in enumerate(lengths):
        ref = _dense_reference(x[b], w, kc[b], vc[b], pos, range(H))
        np.testing.assert_allclose(r["y"][b], ref, rtol=1e-12, atol=1e-12)


def test_single_position_reduces_to_value_projection():
    cfg, w = _block(H=6, KVH=3, seed=7)
    H, KVH, dh = w.H, w.KVH, w.dh
    kc, vc = make_kv_cache(cfg, [0, 0], seed=2)
    x = _x(cfg.d, 2, 5)
    masks = np.array([[0b101101], [0b010010]], np.uint32)
    r = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, masks, kc, vc, [0, 0], H, KVH, dh)
    W, bq, Wo, bo = _f(w.wqkv), _f(w.bqkv), _f(w.wot), _f(w.bo)
    for b in range(2):
        v = (W[(H + KVH) * dh:] @ _f(x[b]) + bq[(H + KVH) * dh:]).astype(np.float16).astype(np.float64)
        y = bo.copy()
        for h in range(H):
            if (int(masks[b, 0]) >> h) & 1:
                g = h // (H // KVH)
                y += Wo[h * dh:(h + 1) * dh].T @ v[g * dh:(g + 1) * dh]
        np.testing.assert_allclose(r["y"][b], y, rtol=1e-12, atol=1e-12)


def test_grouped_heads_equal_repeated_multi_head():
    cfg, w = _block(H=6, KVH=2, seed=11)
    H, KVH, dh, d = w.H, w.KVH, w.dh, w.d
    G = H // KVH
    lengths = [9, 3]
    kc, vc = make_kv_cache(cfg, lengths, seed=4)
    x = _x(d, 2, 8)
    masks = np.array([[0b110101], [0b011110]], np.uint32)
    r = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, masks, kc, vc, lengths, H, KVH, dh)
    # the same block with every KV head repeated for each query head of its group
    rows = w.wqkv.reshape(H + 2 * KVH, dh, d)
    brows = w.bqkv.reshape(H + 2 * KVH, dh)
    rep = [h // G for h in range(H)]
    wq = torch.cat([rows[:H], rows[H:H + KVH][rep], rows[H + KVH:][rep]]).reshape(-1, d)
    bq = torch.cat([brows[:H], brows[H:H + KVH][rep], brows[H + KVH:][rep]]).reshape(-1)
    r2 = oracle.attn_heads(x, wq, bq, w.wot, w.bo, masks, kc[:, rep], vc[:, rep], lengths, H, H, dh)
    np.testing.assert_array_equal(r["y"], r2["y"])
    np.testing.assert_array_equal(r["o"], r2["o"])


def test_no_head_active_gives_bias_and_still_fills_cache():
    cfg, w = _block(H=4, KVH=4, seed=13)
    lengths = [6]
    kc, vc = make_kv_cache(cfg, lengths, seed=5)
    x = _x(cfg.d, 1, 9)
    r = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, np.zeros((1, 1), np.uint32), kc, vc, lengths, 4, 4,
                          cfg.head_dim)
    np.testing.assert_array_equal(r["y"][0], _f(w.bo))
    assert not r["o"].any()
    full = oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, _mask_all(4, 1), kc, vc, lengths, 4, 4,
                             cfg.head_dim)
    np.testing.assert_array_equal(r["kcache"], full["kcache"])
    np.testing.assert_array_equal(r["vcache"], full["vcache"])
    assert (_f(r["kcache"])[0, :, 6] != 0).any()
    np.testing.assert_array_equal(r["kcache"][0, :, :6], kc.numpy().view(np.uint16)[0, :, :6])


def test_head_mask_is_strict_threshold_of_predictor_scores():
    cfg, w = _block(H=12, KVH=12, d=96, seed=17)
    P1, P2, bp = _f(w.p1), _f(w.p2), _f(w.bp)
    hits = 0
    for t in range(8):
        x = _x(cfg.d, 1, 100 + t)[0]
        pr = oracle.attn_predict(x, w.p1, w.p2, w.bp, tau=cfg.tau)
        s = P2 @ (P1 @ _f(x)) + bp
        for h in range(w.H):
            bit = (int(pr["mask"][h // 32]) >> (h % 32)) & 1
            if abs(s[h] - cfg.tau) > 1e-9:
                assert bit == int(s[h] > cfg.tau)
                hits += bit
    assert hits > 0


def test_rejects_bad_arguments():
    cfg, w = _block(H=4, KVH=4, seed=19)
    kc, vc = make_kv_cache(cfg, [2], seed=6)
    x = _x(cfg.d, 1, 1)
    with pytest.raises(ValueError):
        oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, _mask_all(4, 1), kc, vc, [cfg.max_seq], 4, 4,
                          cfg.head_dim)
    with pytest.raises(ValueError):
        oracle.attn_heads(x, w.wqkv, w.bqkv, w.wot, w.bo, _mask_all(4, 1), kc, vc, [2], 4, 3, cfg.head_dim)
