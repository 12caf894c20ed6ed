"""Lookahead predictor on a small synthetic stack: its masks come from the
library's pi_predict with P1' = P1_{l+1} M on layer l's input, and must match
the oracle's predictor run with the same P1' (outside the rounding band); the
reported recalls are checked against a recount on the same tokens."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import mask_matches

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_lookahead_masks_match_oracle_and_report_is_consistent():
    import activation_sparse_ffn_layer_gb300 as P
    from activation_sparse_ffn_layer_gb300 import lookahead as LA
    P.lib()
    cfg = small(CONFIGS["c2"], d=256, F=1024, rank=32, layers=2)
    layers = [make_layer(cfg, l, device=DEV) for l in range(2)]
    n_fit, n_test = 768, 16
    toks = make_tokens(cfg, 0, n_fit + n_test, device=DEV)
    xin = LA.layer_inputs(layers, toks, cfg.tau, cfg.rms_eps)
    x0, x1 = xin[0], xin[1]
    M = LA.fit_map(x0[:n_fit].T.float(), x1[:n_fit].T.float())
    nxt = layers[1]
    p1_look = (nxt.p1.double() @ M).to(torch.float16).contiguous()
    desc_of = lambda nb: P.desc_of(nxt.d, nxt.F, nxt.r, nb, nxt.int4, nxt.gated)
    look = LA._masks(desc_of, x0[n_fit:].contiguous(), p1_look, nxt.p2, nxt.b1, cfg.tau, nxt.F)
    host = oracle.host_layer(dataclasses.replace(nxt, p1=p1_look).to("cpu"))
    W = (nxt.F + 31) // 32
    for t in range(4):
        bits = look[t].cpu().numpy()
        words = np.zeros(W, dtype=np.uint32)
        for k in np.nonzero(bits)[0]:
            words[k // 32] |= np.uint32(1) << np.uint32(k % 32)
        mask_matches(words, oracle.predict(x0[n_fit + t].cpu(), host, cfg.tau), nxt.F, cfg.tau,
                     f"lookahead token {t}")
    rep = LA.evaluate(cfg, 0, n_fit, n_test, device=DEV)
    assert 0.0 < rep.active < 1.0
    assert 0.0 <= rep.recall_lookahead <= 1.0 and 0.0 < rep.recall_standard <= 1.0
    assert 0.0 <= rep.shared <= 1.0
