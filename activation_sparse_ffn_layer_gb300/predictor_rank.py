"""Per-layer predictor sizing on synthetic inputs.

PowerInfer summary (CSDN), section "Adaptive sparse predictor": every layer
gets its own predictor size; for a layer whose activations are skewed the
size is lowered step by step while the predictor still finds at least 95 % of
the neurons that really fire.  Here the predictor is the low-rank linear map
``mask = (P2 (P1 x) + b1 > tau)`` with ``P1 = V_r^T``, ``P2 = U_r S_r`` from a
truncated SVD of the layer's FC1 weights, so its size is the rank r; this
module picks, per layer, the smallest rank (a multiple of ``step``) whose
recall on a set of tokens reaches the target.

All masks and FC1 outputs come from the library's kernels (``pi_predict`` and
``pi_sparse_fc1`` over every row), so the recall is measured on exactly the
arithmetic the decode path runs.  The factorisation is a one-off library call
(``torch.svd_lowrank``), not part of the decode path.

    python -m activation_sparse_ffn_layer_gb300.predictor_rank --config c2 --layers 2
"""
from __future__ import annotations

import argparse
import json
from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import torch

from . import binding as B


@dataclass
class RankChoice:
    rank: int            # chosen rank (max_rank when no candidate reaches the target)
    recall: float        # recall at the chosen rank
    predicted: float     # fraction of (token, neuron) pairs the predictor marks at that rank
    active: float        # fraction of (token, neuron) pairs whose FC1 output is non-zero
    tried: List[tuple]   # (rank, recall) of every candidate evaluated, in order
    reached: bool        # the target was reached


def smallest_rank(recall_of: Callable[[int], float], candidates: Sequence[int], target: float):
    """The first candidate (ascending) whose recall reaches the target.

    Recall need not grow monotonically with the rank, so the candidates are
    scanned in order rather than bisected.  Returns (rank, tried, reached); if
    none reaches the target the largest candidate is returned."""
    tried = []
    for r in sorted(candidates):
        rec = float(recall_of(r))
        tried.append((r, rec))
        if rec >= target:
            return r, tried, True
    return max(candidates), tried, False


def _fc1_weights_fp32(w) -> torch.Tensor:
    """FC1 (gate) rows in storage order as fp32.  INT4 layers carry the
    generator's own reconstruction (codes times group scales), made with
    ``make_layer(..., keep_recon=True)``."""
    if not w.int4:
        return w.w1.float()
    if w.w1_recon is None:
        raise ValueError("INT4 layer without its FC1 reconstruction: build it with make_layer(keep_recon=True)")
    return w.w1_recon


def _unpack(mask: torch.Tensor, F: int) -> torch.Tensor:
    """[T, W] int32 mask words -> [T, F] bool (bit k of word k // 32)."""
    words = mask.to(torch.int64) & 0xFFFFFFFF
    bits = (words.unsqueeze(-1) >> torch.arange(32, device=mask.device)) & 1
    return bits.reshape(mask.shape[0], -1)[:, :F].bool()


class LayerSizer:
    """Recall of rank-r predictors of one layer on a fixed set of tokens."""

    def __init__(self, w, tokens: torch.Tensor, tau: float, max_rank: int, batch: int = 16, seed: int = 0):
        self.w, self.tau, self.batch = w, float(tau), batch
        self.x = tokens.to(torch.float16).contiguous()
        self.T = self.x.shape[0]
        W1 = _fc1_weights_fp32(w)
        q = min(max_rank, w.d, w.F)
        devs = [W1.device] if W1.is_cuda else []
        with torch.random.fork_rng(devices=devs):   # seeded, leaves the caller's generators alone
            torch.manual_seed(seed)
            U, S, V = torch.svd_lowrank(W1, q=q, niter=3)
        self.U, self.S, self.V = U, S, V          # W1 ~= U diag(S) V^T
        self.max_rank = q
        self.truth = self._true_activity()

    def _true_activity(self) -> torch.Tensor:
        """[T, F] bool: FC1 output non-zero, from pi_sparse_fc1 over every row."""
        w, F = self.w, self.w.F
        idx = torch.arange(F, dtype=torch.int32, device=self.x.device)
        cnt = torch.tensor([F], dtype=torch.int32, device=self.x.device)
        ws_struct = B.weights_struct(w)
        out = []
        for t0 in range(0, self.T, self.batch):
            xb = self.x[t0:t0 + self.batch].contiguous()
            nb = xb.shape[0]
            desc = B.desc_of(w.d, F, w.r, nb, w.int4, w.gated)
            ws = torch.zeros(B.pi_workspace_bytes(desc), dtype=torch.uint8, device=self.x.device)
            h = torch.empty(F * nb, dtype=torch.float32, device=self.x.device)
            B.pi_sparse_fc1(desc, xb, ws_struct, idx, cnt, None, h, ws)
            out.append(h.view(F, nb).t() != 0)
        return torch.cat(out, 0)

    def predictor(self, r: int):
        p1 = self.V[:, :r].t().contiguous().to(torch.float16)              # [r, d]
        p2 = (self.U[:, :r] * self.S[:r]).contiguous().to(torch.float16)   # [F, r]
        return p1, p2

    def masks(self, r: int) -> torch.Tensor:
        w, F = self.w, self.w.F
        p1, p2 = self.predictor(r)
        Wd = (F + 31) // 32
        out = []
        for t0 in range(0, self.T, self.batch):
            xb = self.x[t0:t0 + self.batch].contiguous()
            nb = xb.shape[0]
            desc = B.desc_of(w.d, F, r, nb, w.int4, w.gated)
            ws = torch.zeros(B.pi_workspace_bytes(desc), dtype=torch.uint8, device=self.x.device)
            m = torch.zeros(nb, Wd, dtype=torch.int32, device=self.x.device)
            B.pi_predict(desc, xb, p1, p2, w.b1, self.tau, m, ws)
            out.append(_unpack(m, F))
        return torch.cat(out, 0)

    def recall(self, r: int) -> float:
        pred = self.masks(r)
        hit = (pred & self.truth).sum().item()
        return hit / max(1, int(self.truth.sum().item()))

    def choose(self, target: float = 0.95, step: int = 16, min_rank: Optional[int] = None,
               relative: bool = False) -> RankChoice:
        """Smallest candidate rank whose recall reaches `target` (with `relative`,
        `target` times the recall of the largest rank)."""
        lo = min_rank or step
        cands = list(range(lo, self.max_rank + 1, step)) or [self.max_rank]
        if relative:
            target = target * self.recall(self.max_rank)
        r, tried, reached = smallest_rank(self.recall, cands, target)
        pred = self.masks(r)
        return RankChoice(rank=r, recall=dict(tried).get(r, self.recall(r)),
                          predicted=float(pred.float().mean().item()),
                          active=float(self.truth.float().mean().item()), tried=tried, reached=reached)


def main(argv=None):
    from synth import CONFIGS, make_layer, make_tokens

    ap = argparse.ArgumentParser(description="smallest predictor rank per layer with recall >= target")
    ap.add_argument("--config", default="c2")
    ap.add_argument("--layers", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=64)
    ap.add_argument("--target", type=float, default=0.95)
    ap.add_argument("--step", type=int, default=16)
    ap.add_argument("--relative", action="store_true",
                    help="target is a fraction of the recall at the configured rank")
    args = ap.parse_args(argv)
    assert torch.cuda.is_available(), "needs a CUDA GPU"
    B.lib()
    cfg = CONFIGS[args.config]
    x = make_tokens(cfg, 0, args.tokens, device="cuda")
    for l in range(args.layers):
        w = make_layer(cfg, l, device="cuda", keep_recon=True)
        ch = LayerSizer(w, x, cfg.tau, max_rank=cfg.layer_rank(l)).choose(args.target, args.step,
                                                                          relative=args.relative)
        pred_bytes = 2 * ch.rank * (cfg.d + cfg.F)
        print(json.dumps({"layer": l, "rank": ch.rank, "configured_rank": cfg.layer_rank(l),
                          "recall": round(ch.recall, 4), "predicted": round(ch.predicted, 4),
                          "active": round(ch.active, 4), "reached": ch.reached,
                          "predictor_MB": round(pred_bytes / 1e6, 2),
                          "tried": [(r, round(v, 4)) for r, v in ch.tried]}), flush=True)


if __name__ == "__main__":
    main()
