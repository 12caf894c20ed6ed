"""Pins of the oracle's FFN functions (dense, masked, FC1/FC2, gated, INT4, norm).

- the dense FFN equals torch's Linear -> ReLU -> Linear in fp64 (library);
- invariant (i): a mask that contains every neuron the ReLU keeps gives the
  dense output; a mask holding none of them gives b2 exactly (PowerInfer
  summary (CSDN), section "Background": only neurons with positive FC1 output
  contribute to FC2);
- invariant (ii): permuting the neuron table (and the stored rows with it)
  leaves the output bit-identical (section "Neuron placement and management");
- invariant (iii): brute force over all 2^F masks of a tiny layer: every
  mask's contribution is the sum of its single neurons' contributions;
- gated and INT4 layers reduce, in special cases, to the plain fp16 layer;
- FC1, FC2 and the gated FC1 against a layer worked by hand
  (tests/golden/ffn_small.txt); the gated layer in general against torch's
  products in fp64;
- the normalisation against hand-worked values and its guard band.
"""
import itertools
import os
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dense_torch(x, w1, b1, w2t, b2):
    f1 = torch.nn.Linear(w1.shape[1], w1.shape[0]).double()
    f2 = torch.nn.Linear(w1.shape[0], w1.shape[1]).double()
    with torch.no_grad():
        f1.weight.copy_(torch.from_numpy(w1.astype(np.float64)))
        f1.bias.copy_(torch.from_numpy(b1.astype(np.float64)))
        f2.weight.copy_(torch.from_numpy(w2t.astype(np.float64).T))
        f2.bias.copy_(torch.from_numpy(b2.astype(np.float64)))
        y = torch.nn.Sequential(f1, torch.nn.ReLU(), f2)(torch.from_numpy(x.astype(np.float64)))
    return y.numpy()


def _np16(t):
    return t.numpy() if hasattr(t, "numpy") else t


def _mask_from_bits(bits):
    F = len(bits)
    m = np.zeros((F + 31) // 32, np.uint32)
    for k, b in enumerate(bits):
        if b:
            m[k // 32] |= np.uint32(1 << (k % 32))
    return m


@pytest.fixture(scope="module")
def layer_small():
    cfg = small(CONFIGS["c1"], d=128, F=256, rank=16)
    return cfg, make_layer(cfg, 0), make_tokens(cfg, 0, 3)


def test_dense_matches_torch_mlp(layer_small):
    cfg, w, xs = layer_small
    for t in range(3):
        y = oracle.ffn_dense(xs[t], w)
        ref = _dense_torch(_np16(xs[t]), _np16(w.w1), _np16(w.b1), _np16(w.w2t), _np16(w.b2))
        np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_masked_superset_equals_dense(layer_small):
    cfg, w, xs = layer_small
    rng = np.random.default_rng(6)
    for t in range(3):
        x = xs[t]
        h = oracle.fc1(x, w, np.arange(cfg.F, dtype=np.int32))
        active = h > 0
        dense = oracle.ffn_dense(x, w)
        full = oracle.ffn_masked(x, w, _mask_from_bits(np.ones(cfg.F, bool)))
        exact = oracle.ffn_masked(x, w, _mask_from_bits(active))
        sup = oracle.ffn_masked(x, w, _mask_from_bits(active | (rng.random(cfg.F) < 0.3)))
        for y in (full, exact, sup):
            np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-14)
        b2 = _np16(w.b2).astype(np.float64)
        assert np.array_equal(oracle.ffn_masked(x, w, _mask_from_bits(~active)), b2)
        assert np.array_equal(oracle.ffn_masked(x, w, _mask_from_bits(np.zeros(cfg.F, bool))), b2)
        # dropping one neuron the ReLU keeps must change the result
        k = int(np.nonzero(active)[0][0])
        drop = active.copy(); drop[k] = False
        assert not np.allclose(oracle.ffn_masked(x, w, _mask_from_bits(drop)), dense, rtol=1e-9, atol=0)


def test_table_permutation_invariance():
    cfg = small(CONFIGS["c1"], d=64, F=96, rank=8)
    w_hot = make_layer(cfg, 0)
    perm = torch.from_numpy(np.random.default_rng(7).permutation(cfg.F).astype(np.int32))
    w_perm = make_layer(cfg, 0, table_override=perm)
    x = make_tokens(cfg, 0, 1)[0]
    chosen = set(np.random.default_rng(8).choice(cfg.F, 30, replace=False).tolist())  # original ids
    outs = []
    for w in (w_hot, w_perm):
        tb = w.table.numpy()
        outs.append(oracle.ffn_masked(x, w, _mask_from_bits([int(o) in chosen for o in tb])))
    assert np.array_equal(outs[0], outs[1])
    # and the rows really were stored in a different order
    assert not np.array_equal(w_hot.table.numpy(), w_perm.table.numpy())


def test_bruteforce_all_masks_tiny_layer():
    rng = np.random.default_rng(9)
    d, F = 6, 10
    L = SimpleNamespace(d=d, F=F, r=1, gated=False, int4=False,
                        w1=(rng.standard_normal((F, d))).astype(np.float16),
                        b1=(rng.standard_normal(F)).astype(np.float16),
                        w2t=(rng.standard_normal((F, d))).astype(np.float16),
                        b2=(rng.standard_normal(d)).astype(np.float16),
                        p1=np.zeros((1, d), np.float16), p2=np.zeros((F, 1), np.float16),
                        table=rng.permutation(F).astype(np.int32), wu=None)
    H = oracle.host_layer(L)
    x = rng.standard_normal(d).astype(np.float16)
    b2 = L.b2.astype(np.float64)
    single = [oracle.ffn_masked(x, H, _mask_from_bits([j == k for j in range(F)])) - b2 for k in range(F)]
    for bits in itertools.product((False, True), repeat=F):
        y = oracle.ffn_masked(x, H, _mask_from_bits(bits))
        want = b2 + sum((single[k] for k in range(F) if bits[k]), np.zeros(d))
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)
    # the dense output is the all-ones mask
    np.testing.assert_allclose(oracle.ffn_masked(x, H, _mask_from_bits([True] * F)),
                               oracle.ffn_dense(x, H), rtol=1e-13, atol=1e-13)


def test_fc1_fc2_compose_to_masked(layer_small):
    cfg, w, xs = layer_small
    x = xs[0]
    pr = oracle.predict(x, w, cfg.tau)
    idx, _, n = oracle.compact(pr["mask"], cfg.F, w.table)
    assert n > 0
    y = oracle.fc2(oracle.fc1(x, w, idx), w, idx)
    np.testing.assert_allclose(y, oracle.ffn_masked(x, w, pr["mask"]), rtol=1e-12, atol=1e-14)


def test_gated_with_unit_up_projection_is_plain_relu():
    rng = np.random.default_rng(10)
    d, F = 32, 48
    wg = (rng.standard_normal((F, d)) * 0.2).astype(np.float16)
    wu = np.zeros((F, d), np.float16); wu[:, 0] = 1            # Wu x = x_0 = 1 exactly
    x = rng.standard_normal(d).astype(np.float16); x[0] = 1
    common = dict(d=d, F=F, r=1, int4=False, w1=wg, b1=(rng.standard_normal(F) * 0.3).astype(np.float16),
                  w2t=(rng.standard_normal((F, d)) * 0.2).astype(np.float16),
                  b2=np.zeros(d, np.float16), p1=np.zeros((1, d), np.float16),
                  p2=np.zeros((F, 1), np.float16), table=np.arange(F, dtype=np.int32))
    gated = SimpleNamespace(gated=True, wu=wu, **common)
    plain = SimpleNamespace(gated=False, wu=None, **common)
    assert np.array_equal(oracle.ffn_dense(x, gated), oracle.ffn_dense(x, plain))
    # and a scaled up projection scales each neuron's output: Wu x = 2 -> y - b2 doubles
    wu2 = wu.copy(); wu2[:, 0] = 2
    g2 = SimpleNamespace(gated=True, wu=wu2, **common)
    np.testing.assert_allclose(oracle.ffn_dense(x, g2), 2 * oracle.ffn_dense(x, plain), rtol=1e-13)


def test_int4_layer_equals_fp16_layer_with_same_values():
    # power-of-two scales make every q*s exactly representable in binary16, so
    # the INT4 layer and the fp16 layer holding the decoded values must agree bit for bit
    rng = np.random.default_rng(11)
    d, F = 64, 40
    def pack(codes):
        out = np.zeros((codes.shape[0], codes.shape[1] // 2), np.uint8)
        for c in range(codes.shape[1]):
            out[:, c // 2] |= ((codes[:, c] & 0xF) << (4 * (c % 2))).astype(np.uint8)
        return out
    q1, q2 = rng.integers(-8, 8, (F, d)), rng.integers(-8, 8, (F, d))
    s1 = (2.0 ** rng.integers(-9, -5, (F, d // 32))).astype(np.float16)
    s2 = (2.0 ** rng.integers(-9, -5, (F, d // 32))).astype(np.float16)
    w1 = (q1 * np.repeat(s1.astype(np.float64), 32, axis=1)).astype(np.float16)
    w2t = (q2 * np.repeat(s2.astype(np.float64), 32, axis=1)).astype(np.float16)
    common = dict(d=d, F=F, r=1, gated=False, wu=None, b1=(rng.standard_normal(F) * 0.1).astype(np.float16),
                  b2=(rng.standard_normal(d) * 0.1).astype(np.float16), p1=np.zeros((1, d), np.float16),
                  p2=np.zeros((F, 1), np.float16), table=rng.permutation(F).astype(np.int32))
    L4 = SimpleNamespace(int4=True, w1_q=pack(q1), w1_s=s1, w2t_q=pack(q2), w2t_s=s2, **common)
    L16 = SimpleNamespace(int4=False, w1=w1, w2t=w2t, **common)
    x = rng.standard_normal(d).astype(np.float16)
    mask = _mask_from_bits(rng.random(F) < 0.5)
    assert np.array_equal(oracle.ffn_masked(x, L4, mask), oracle.ffn_masked(x, L16, mask))
    assert np.array_equal(oracle.ffn_dense(x, L4), oracle.ffn_dense(x, L16))


def test_rmsnorm_hand_examples():
    with open(os.path.join(GOLDEN, "rmsnorm_small.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            _, ys, bits = line.split()
            y = np.array([float(v) for v in ys.split(",")])
            want = [int(b, 16) for b in bits.split(",")]
            xb, _, _ = oracle.rmsnorm_half(y, 1e-6)
            assert xb.tolist() == want, (ys, [hex(v) for v in xb])


def test_rmsnorm_band_bounds_fp32_evaluation():
    rng = np.random.default_rng(12)
    for d in (7, 768, 4096):
        y = rng.standard_normal(d) * 0.3
        _, pre, band = oracle.rmsnorm_half(y, 1e-6)
        y32 = y.astype(np.float32)
        for ss in (np.sum(y32 * y32, dtype=np.float32),
                   np.float32(sum(float(np.float32(v * v)) for v in y32[::-1]))):
            scale = np.float32(1.0) / np.sqrt(np.float32(ss / np.float32(d)) + np.float32(1e-6))
            v32 = (y32 * scale).astype(np.float64)
            # the fp64 pre-rounding value of the float32 input
            _, pre32, _ = oracle.rmsnorm_half(y32.astype(np.float64), 1e-6)
            assert np.all(np.abs(v32 - pre32) <= band / 2 + 1e-300)


def _fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out.setdefault(k, []).append([float(t) for t in v])
    return out


def _hand_layer(g, gated):
    h16 = lambda rows: np.asarray(rows, dtype=np.float64).astype(np.float16)
    F = len(g["w1"])
    d = len(g["x"][0])
    return SimpleNamespace(d=d, F=F, r=1, int4=False, gated=gated, w1=h16(g["w1"]), b1=h16(g["b1"][0]),
                           wu=h16(g["wu"]) if gated else None, w2t=h16(g["w2t"]), b2=h16(g["b2"][0]),
                           p1=np.zeros((1, d), np.float16), p2=np.zeros((F, 1), np.float16),
                           table=np.arange(F, dtype=np.int32))


def test_fc1_fc2_hand_example():
    g = _fixture("ffn_small.txt")
    x = np.asarray(g["x"][0], dtype=np.float64).astype(np.float16)
    for gated, hk, yk in ((False, "h", "y"), (True, "h_gated", "y_gated")):
        L = _hand_layer(g, gated)
        idx = np.arange(L.F, dtype=np.int32)
        h = oracle.fc1(x, L, idx)
        np.testing.assert_array_equal(h, g[hk][0])
        np.testing.assert_array_equal(oracle.fc2(h, L, idx), g[yk][0])
        np.testing.assert_array_equal(oracle.ffn_dense(x, L), g[yk][0])
        np.testing.assert_array_equal(oracle.ffn_masked(x, L, _mask_from_bits([True] * L.F)), g[yk][0])
    L = _hand_layer(g, False)
    idx = np.asarray(g["fc2_idx"][0], dtype=np.int32)
    np.testing.assert_array_equal(oracle.fc2(np.asarray(g["fc2_h"][0]), L, idx), g["fc2_y"][0])
    # FC1 on a sub-list returns the listed rows' outputs in list order
    np.testing.assert_array_equal(oracle.fc1(x, L, np.asarray([2, 1], np.int32)), [0.0, 0.5])


def test_gated_layer_matches_torch_products():
    rng = np.random.default_rng(21)
    d, F = 48, 40
    wg = (rng.standard_normal((F, d)) * 0.2).astype(np.float16)
    wu = (rng.standard_normal((F, d)) * 0.2).astype(np.float16)
    w2t = (rng.standard_normal((F, d)) * 0.2).astype(np.float16)
    bg = (rng.standard_normal(F) * 0.3).astype(np.float16)
    b2 = (rng.standard_normal(d) * 0.1).astype(np.float16)
    x = rng.standard_normal(d).astype(np.float16)
    L = SimpleNamespace(d=d, F=F, r=1, int4=False, gated=True, w1=wg, b1=bg, wu=wu, w2t=w2t, b2=b2,
                        p1=np.zeros((1, d), np.float16), p2=np.zeros((F, 1), np.float16),
                        table=np.arange(F, dtype=np.int32))
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    gate = torch.nn.functional.linear(t(x), t(wg), t(bg))
    up = torch.nn.functional.linear(t(x), t(wu))
    h = torch.relu(gate) * up
    y = torch.nn.functional.linear(h, t(w2t).T, t(b2))
    np.testing.assert_allclose(oracle.fc1(x, L, np.arange(F, dtype=np.int32)), h.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.ffn_dense(x, L), y.numpy(), rtol=1e-12, atol=1e-13)
    assert 0 < int((h.numpy() != 0).sum()) < F
