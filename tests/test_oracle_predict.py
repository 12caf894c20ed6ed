"""Pins of the oracle's predictor, mask layout and compaction.

- a predictor worked by hand (tests/golden/predict_small.txt);
- the special case P1 = I, P2 = W1, tau = 0, where the predicted set must be
  exactly the set of neurons the FFN's ReLU keeps (checked through the
  oracle's separate FFN code);
- the guard band really bounds fp32 evaluations of the score;
- compaction against hand-worked masks and against its defining properties;
- the batch union of masks against a hand-worked example (tests/golden/mask_union_small.txt).
"""
import os
from types import SimpleNamespace

import numpy as np

import oracle
from synth import CONFIGS, make_layer, make_tokens, small

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


def _layer(**kw):
    base = dict(gated=False, int4=False, wu=None, table=None)
    base.update(kw)
    L = SimpleNamespace(**base)
    if L.table is None:
        L.table = np.arange(L.F, dtype=np.int32)
    return L


def test_predict_hand_example():
    g = _fixture("predict_small.txt")
    x = np.array(g["x"][0], np.float16)
    p1 = np.array(g["p1"], np.float16)
    p2 = np.array(g["p2"], np.float16)
    b = np.array(g["b"][0], np.float16)
    L = _layer(d=4, F=6, r=2, p1=p1, p2=p2, b1=b, w1=np.zeros((6, 4), np.float16),
               w2t=np.zeros((6, 4), np.float16), b2=np.zeros(4, np.float16))
    for tau, word in g["mask"]:
        out = oracle.predict(x, L, tau)
        assert np.array_equal(out["u"], np.array(g["u"][0]))
        assert np.array_equal(out["s"], np.array(g["s"][0]))
        assert int(out["mask"][0]) == int(word), (tau, out["mask"])


def test_mask_bit_layout_spans_words():
    # F = 70: three words; make exactly neurons 1, 33 and 69 score above tau
    F, d, r = 70, 8, 1
    p1 = np.zeros((r, d), np.float16); p1[0, 0] = 1
    p2 = np.zeros((F, r), np.float16)
    b = np.full(F, -1, np.float16)
    for k in (1, 33, 69):
        p2[k, 0] = 2
    x = np.zeros(d, np.float16); x[0] = 1
    L = _layer(d=d, F=F, r=r, p1=p1, p2=p2, b1=b, w1=np.zeros((F, d), np.float16),
               w2t=np.zeros((F, d), np.float16), b2=np.zeros(d, np.float16))
    m = oracle.predict(x, L, 0.0)["mask"]
    assert m.tolist() == [1 << 1, 1 << 1, 1 << 5]


def test_identity_predictor_predicts_exactly_the_relu_set():
    # P1 = I, P2 = W1, bias = b1 -> s = W1 x + b1 = z.  With tau = 0 the mask
    # must be the set where the FFN's ReLU output is positive.
    rng = np.random.default_rng(3)
    d, F = 16, 80
    w1 = (rng.standard_normal((F, d)) * 0.25).astype(np.float16)
    b1 = (rng.standard_normal(F) * 0.5).astype(np.float16)
    L = _layer(d=d, F=F, r=d, p1=np.eye(d, dtype=np.float16), p2=w1, b1=b1, w1=w1,
               w2t=np.zeros((F, d), np.float16), b2=np.zeros(d, np.float16))
    for t in range(5):
        x = rng.standard_normal(d).astype(np.float16)
        mask = oracle.predict(x, L, 0.0)["mask"]
        h = oracle.fc1(x, L, np.arange(F, dtype=np.int32))
        bits = np.array([(mask[k // 32] >> (k % 32)) & 1 for k in range(F)])
        assert np.array_equal(bits == 1, h > 0)


def test_guard_band_bounds_fp32_scores():
    cfg = small(CONFIGS["c1"], d=256, F=512, rank=32)
    w = make_layer(cfg, 0)
    x = make_tokens(cfg, 0, 3)
    p1 = w.p1.float().numpy().astype(np.float32)
    p2 = w.p2.float().numpy().astype(np.float32)
    b = w.b1.float().numpy().astype(np.float32)
    for t in range(3):
        out = oracle.predict(x[t], w, cfg.tau)
        xf = x[t].float().numpy().astype(np.float32)
        evals = []
        u32 = np.zeros(cfg.rank, np.float32)
        for j in range(cfg.d):                      # sequential fp32 sums, forward
            u32 += p1[:, j] * xf[j]
        s32 = b.copy()
        for i in range(cfg.rank):
            s32 += p2[:, i] * u32[i]
        evals.append(s32)
        u32 = np.zeros(cfg.rank, np.float32)        # backward
        for j in reversed(range(cfg.d)):
            u32 += p1[:, j] * xf[j]
        s32 = np.zeros(cfg.F, np.float32)
        for i in reversed(range(cfg.rank)):
            s32 += p2[:, i] * u32[i]
        evals.append(s32 + b)
        evals.append((p2 @ (p1 @ xf)) + b)          # BLAS blocking
        for s32 in evals:
            err = np.abs(s32.astype(np.float64) - out["s"])
            assert np.all(err <= out["band"] / 2), float(np.max(err / out["band"]))


def test_compact_hand_examples():
    idx, orig, n = oracle.compact(np.array([0b1011, 0x80000000], np.uint32), 64,
                                  table=np.arange(64)[::-1].astype(np.int32))
    assert n == 4 and idx.tolist() == [0, 1, 3, 63] and orig.tolist() == [63, 62, 60, 0]
    idx, _, n = oracle.compact(np.zeros(3, np.uint32), 70)
    assert n == 0 and idx.size == 0
    idx, _, n = oracle.compact(np.array([0xFFFFFFFF, 0xFFFFFFFF, 0x3F], np.uint32), 70)
    assert n == 70 and idx.tolist() == list(range(70))


def test_compact_properties_random():
    rng = np.random.default_rng(4)
    for F in (1, 31, 32, 33, 100, 1000, 3001):
        words = (F + 31) // 32
        m = rng.integers(0, 2 ** 32, size=words, dtype=np.uint64).astype(np.uint32)
        if F % 32:
            m[-1] &= np.uint32((1 << (F % 32)) - 1)
        idx, _, n = oracle.compact(m, F)
        assert n == sum(bin(int(v)).count("1") for v in m)
        assert np.all(np.diff(idx) > 0)
        listed = set(idx.tolist())
        for k in range(F):
            assert (((int(m[k // 32]) >> (k % 32)) & 1) == 1) == (k in listed)


def test_worked_example_hot_3_5_7_predicted_3_4_5():
    # PowerInfer summary (CSDN), section "Insights and overview": neurons 3, 5, 7
    # are hot and placed first; the predictor says 3, 4, 5; 3 and 5 are computed
    # from the hot part, 4 from the rest, 7 is skipped.
    F = 8
    table = np.array([3, 5, 7, 0, 1, 2, 4, 6], np.int32)      # storage row -> original id
    predicted = {3, 4, 5}
    mask = np.zeros(1, np.uint32)
    for k in range(F):
        if table[k] in predicted:
            mask[0] |= np.uint32(1 << k)
    idx, orig, n = oracle.compact(mask, F, table)
    assert n == 3
    assert idx.tolist() == [0, 1, 6]
    assert orig.tolist() == [3, 5, 4]
    n_hot = 3
    assert sorted(orig[idx < n_hot].tolist()) == [3, 5]
    assert orig[idx >= n_hot].tolist() == [4]
    assert 7 not in orig.tolist()


def test_mask_union_is_bitwise_or():
    rng = np.random.default_rng(5)
    masks = rng.integers(0, 2 ** 32, size=(5, 4), dtype=np.uint64).astype(np.uint32)
    u = oracle.mask_union(masks, 128)
    for w in range(4):
        acc = 0
        for b in range(5):
            acc |= int(masks[b, w])
        assert int(u[w]) == acc


def test_mask_union_hand_example():
    g = _fixture("mask_union_small.txt")
    F = int(g["F"][0][0])
    masks = np.asarray(g["mask"], dtype=np.uint64).astype(np.uint32)
    u = oracle.mask_union(masks, F)
    assert [int(v) for v in u] == [int(v) for v in g["union"][0]]


def test_guard_band_is_not_vacuous():
    """The band is a worst-case bound (gamma_n times the sums of absolute
    terms), so it is far wider than the error a typical fp32 order makes (on
    these layers about 10^4 times the largest error of a BLAS-blocked
    evaluation); what matters is that it excuses only scores next to the
    threshold: on layers with the workloads' statistics it covers at most
    0.5 % of the neurons."""
    for base, d, F, r in ((CONFIGS["c2"], 1024, 4096, 64), (CONFIGS["c4"], 1024, 4096, 128)):
        cfg = small(base, d=d, F=F, rank=r)
        w = make_layer(cfg, 0)
        xs = make_tokens(cfg, 0, 4)
        p1 = w.p1.float().numpy().astype(np.float32)
        p2 = w.p2.float().numpy().astype(np.float32)
        b = w.b1.float().numpy().astype(np.float32)
        in_band, total = 0, 0
        for t in range(4):
            out = oracle.predict(xs[t], w, cfg.tau)
            in_band += int(np.sum(np.abs(out["s"] - np.float64(np.float32(cfg.tau))) <= out["band"]))
            total += cfg.F
            s32 = (p2 @ (p1 @ xs[t].float().numpy().astype(np.float32))) + b
            assert np.all(np.abs(s32.astype(np.float64) - out["s"]) <= out["band"])
        assert in_band <= 0.005 * total, (base.key, in_band, total)
