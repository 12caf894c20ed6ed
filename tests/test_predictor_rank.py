"""Host logic of the per-layer predictor sizing (no GPU): the candidate scan,
the mask unpacking and the INT4 FC1 rows used for the factorisation (the
generator's reconstruction, pinned against the oracle's own FC1 of the same
packed rows)."""
import numpy as np
import torch

import oracle
from activation_sparse_ffn_layer_gb300.predictor_rank import _fc1_weights_fp32, _unpack, smallest_rank
from synth import CONFIGS, make_layer, make_tokens, small


def test_smallest_rank_scans_in_order():
    rec = {16: 0.80, 32: 0.93, 48: 0.96, 64: 0.99}
    r, tried, ok = smallest_rank(rec.__getitem__, [64, 16, 48, 32], 0.95)
    assert (r, ok) == (48, True) and [t[0] for t in tried] == [16, 32, 48]
    # not monotone: the first candidate that reaches the target wins
    rec2 = {16: 0.96, 32: 0.90, 48: 0.97}
    assert smallest_rank(rec2.__getitem__, [16, 32, 48], 0.95)[0] == 16
    # none reaches it: the largest candidate, flagged
    r, tried, ok = smallest_rank(rec.__getitem__, [16, 32], 0.999)
    assert (r, ok) == (32, False) and len(tried) == 2


def test_unpack_bits():
    words = torch.tensor([[0b1011, -1], [-(1 << 31), 0]], dtype=torch.int32)
    bits = _unpack(words, 40)
    assert bits.shape == (2, 40)
    assert bits[0, :4].tolist() == [True, True, False, True]
    assert bits[0, 32:40].all() and not bits[0, 4:32].any()
    assert bits[1, 31] and bits[1].sum() == 1


def test_int4_decode_matches_oracle_fc1():
    cfg = small(CONFIGS["c5"], d=256, F=96, rank=16)
    w = make_layer(cfg, 0, device="cpu", keep_recon=True)
    x = make_tokens(cfg, 0, 1, device="cpu")[0]
    W = _fc1_weights_fp32(w).double().numpy()
    z = W @ x.double().numpy() + w.b1.double().numpy()
    h_ref = np.maximum(z, 0.0)
    h_or = oracle.fc1(x, w, np.arange(w.F, dtype=np.int32))
    assert np.allclose(h_or, h_ref, rtol=1e-12, atol=1e-12)
