"""Per-layer predictor sizing on the GPU: the chosen rank's recall reaches the
target and the next smaller candidate's does not, and the recall measured from
the library's kernels agrees with the recall of the same rank-r predictor
computed by the fp64 oracle (masks from oracle.predict, activity from
oracle.fc1) on a sample of the tokens."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("kind,cfg", [
    ("fp16", small(CONFIGS["c2"], d=1024, F=4096, rank=96)),
    ("int4", small(CONFIGS["c5"], d=1024, F=4096, rank=96)),
], ids=["fp16", "int4"])
def test_rank_choice_and_oracle_recall(kind, cfg):
    import activation_sparse_ffn_layer_gb300 as P
    from activation_sparse_ffn_layer_gb300.predictor_rank import LayerSizer
    P.lib()
    w = make_layer(cfg, 0, device=DEV, keep_recon=True)
    x = make_tokens(cfg, 0, 32, device=DEV)
    sz = LayerSizer(w, x, cfg.tau, max_rank=cfg.rank)
    ch = sz.choose(target=0.95, step=16)
    tried = dict(ch.tried)
    if ch.reached:
        assert ch.recall >= 0.95
        assert all(v < 0.95 for r, v in ch.tried if r < ch.rank)
    else:
        assert all(v < 0.95 for v in tried.values()) and ch.rank == max(tried)
    assert 0.0 < ch.active < 1.0 and 0.0 < ch.predicted < 1.0
    # the same rank-r predictor in the oracle, on 6 tokens
    p1, p2 = sz.predictor(ch.rank)
    wr = dataclasses.replace(w, p1=p1, p2=p2, r=ch.rank)
    wh = oracle.host_layer(wr.to("cpu"))
    xs = x[:6].cpu()
    allrows = np.arange(w.F, dtype=np.int32)
    hit = act = 0
    for t in range(6):
        m = oracle.predict(xs[t], wh, cfg.tau)["mask"]
        pred = ((m[np.arange(w.F) // 32] >> (np.arange(w.F) % 32)) & 1).astype(bool)
        true = oracle.fc1(xs[t], wh, allrows) > 0
        hit += int((pred & true).sum())
        act += int(true.sum())
    rec_oracle = hit / act
    pred_gpu = sz.masks(ch.rank)[:6].cpu().numpy()
    true_gpu = sz.truth[:6].cpu().numpy()
    rec_gpu = (pred_gpu & true_gpu).sum() / true_gpu.sum()
    assert abs(rec_gpu - rec_oracle) <= 0.01, (rec_gpu, rec_oracle)


def test_relative_target():
    """Relative sizing: the chosen rank keeps at least the requested fraction of
    the recall at the configured rank; every smaller candidate keeps less."""
    import activation_sparse_ffn_layer_gb300 as P
    from activation_sparse_ffn_layer_gb300.predictor_rank import LayerSizer
    P.lib()
    cfg = small(CONFIGS["c2"], d=1024, F=4096, rank=96)
    w = make_layer(cfg, 0, device=DEV)
    sz = LayerSizer(w, make_tokens(cfg, 0, 32, device=DEV), cfg.tau, max_rank=cfg.rank)
    full = sz.recall(cfg.rank)
    ch = sz.choose(target=0.98, step=16, relative=True)
    assert ch.reached and ch.recall >= 0.98 * full
    assert all(v < 0.98 * full for r, v in ch.tried if r < ch.rank)
