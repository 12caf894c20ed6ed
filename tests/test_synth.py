"""Checks of the synthetic workload generator against the statistics it is
meant to reproduce (these check inputs, not the decode path)."""
import math

import numpy as np
import pytest
import torch

from synth import CONFIGS, make_layer, make_tokens, small, zipf_probabilities, predictor_param_share
from synth.generate import _quantize_g32


@pytest.mark.parametrize("key", list(CONFIGS))
def test_predictor_budget_within_ten_percent(key):
    # PowerInfer summary (CSDN), section "Adaptive sparse predictor": predictor
    # parameters are kept within 10% of the model's parameters.
    assert predictor_param_share(CONFIGS[key]) <= 0.10


@pytest.mark.parametrize("F,s,m", [(3072, 1.1, 0.10), (28672, 1.0, 0.12), (49152, 1.1, 0.06)])
def test_zipf_mean_and_shape(F, s, m):
    p = zipf_probabilities(F, s, m)
    assert abs(float(p.mean()) - m) < 1e-9
    assert float(p.max()) <= 0.999 + 1e-12
    assert torch.all(p[:-1] >= p[1:])                   # non-increasing in rank


def test_true_firing_rate_and_table():
    cfg = CONFIGS["c1"]
    w = make_layer(cfg, 0)
    x = make_tokens(cfg, 0, 64).float()
    z = x @ w.w1.float().T + w.b1.float()
    rate = float((z > 0).float().mean())
    assert abs(rate - cfg.mean_rate) < 0.02
    tb = w.table.numpy()
    assert sorted(tb.tolist()) == list(range(cfg.F))
    p = w.p_fire.numpy()[tb]
    n_hot = cfg.n_hot()
    assert np.all(np.diff(p[:n_hot]) <= 0)              # hot prefix by descending probability
    assert np.all(np.diff(tb[n_hot:]) > 0)              # cold part in original order
    assert p[:n_hot].sum() / p.sum() > 0.6


def test_c3_rank_rule():
    cfg = CONFIGS["c3"]
    ranks = [cfg.layer_rank(l) for l in range(cfg.layers)]
    rates = [cfg.layer_rate(l) for l in range(cfg.layers)]
    assert min(ranks) == 64 and max(ranks) == 512 and all(r % 32 == 0 for r in ranks)
    order = np.argsort(rates)
    assert all(ranks[order[i]] <= ranks[order[i + 1]] for i in range(len(order) - 1))
    assert abs(np.mean(rates) - 0.08) < 1e-12


def test_int4_quantiser_codes_in_range_and_packing():
    w = torch.randn(4, 64) * 0.02
    packed, s, recon = _quantize_g32(w)
    assert packed.shape == (4, 32) and s.shape == (4, 2) and s.dtype == torch.float16
    lo = (packed & 0xF).to(torch.int16)
    hi = (packed >> 4).to(torch.int16)
    lo = torch.where(lo >= 8, lo - 16, lo)
    hi = torch.where(hi >= 8, hi - 16, hi)
    codes = torch.stack([lo, hi], 2).reshape(4, 64)
    assert int(codes.min()) >= -8 and int(codes.max()) <= 7
    assert torch.equal(codes.float() * s.float().repeat_interleave(32, 1), recon)
    assert float((recon - w).abs().max()) <= float(s.float().max()) * 0.51


def test_same_seed_same_layer():
    cfg = small(CONFIGS["c2"], d=64, F=128, rank=8)
    a, b = make_layer(cfg, 3), make_layer(cfg, 3)
    for k, t in a.tensors().items():
        assert torch.equal(t, b.tensors()[k]), k
    assert not torch.equal(a.w1, make_layer(cfg, 4).w1)
