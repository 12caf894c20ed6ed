"""Lookahead prediction: layer l+1's active neurons from layer l's input.

The PowerInfer summary (CSDN), section "Background", notes that which neurons
of a layer fire can be foreseen a few layers ahead, which lets a system fetch
those neurons before the layer runs.  This module builds such a lookahead
predictor for the synthetic stacks and measures it; it does not change what
the decode path computes (the layer's own predictor still decides its mask).

Construction (no training data: fitted on synthetic decode tokens):

* run N seeded tokens through layers l and l+1 with the library's stack call
  and keep each token's input to both layers (x_l, x_{l+1});
* fit the linear map M that best carries x_l to x_{l+1} in the least-squares
  sense, with a small ridge term: M = X1 X0^T (X0 X0^T + lam I)^-1;
* the lookahead predictor of layer l+1 is layer l+1's own low-rank predictor
  composed with M: P1' = P1_{l+1} M (rank r, the same shape and cost as
  P1), P2' = P2_{l+1}, bias b1_{l+1}.  Its mask for token t is taken by the
  library's pi_predict on x_l.

Reported on held-out tokens: the recall of the neurons whose FC1 output is
non-zero (from pi_sparse_fc1 over every row) for the standard predictor (on
x_{l+1}) and for the lookahead one (on x_l), and the share of the standard
predictor's rows that the lookahead one also names (the rows a one-layer-early
prefetch would have fetched).

    python -m activation_sparse_ffn_layer_gb300.lookahead --config c2 --layer 0 --fit 8192 --test 64
"""
from __future__ import annotations

import argparse
import dataclasses
import json

import torch

from . import binding as B


def fit_map(X0: torch.Tensor, X1: torch.Tensor, lam: float = 1e-3) -> torch.Tensor:
    """Least-squares linear map M (d x d) with X1 ~= M X0, columns = tokens:
    M = X1 X0^T (X0 X0^T + lam * tr(X0 X0^T) / d * I)^-1, in fp64."""
    X0 = X0.double()
    X1 = X1.double()
    d = X0.shape[0]
    G = X0 @ X0.T
    reg = lam * torch.trace(G) / d
    G = G + reg * torch.eye(d, dtype=G.dtype, device=G.device)
    C = X1 @ X0.T
    # M G = C  ->  M = C G^-1 (G symmetric positive definite)
    return torch.linalg.solve(G, C.T).T


def _unpack(mask: torch.Tensor, F: int) -> torch.Tensor:
    words = mask.to(torch.int64) & 0xFFFFFFFF
    bits = (words.unsqueeze(-1) >> torch.arange(32, device=mask.device)) & 1
    return bits.reshape(mask.shape[0], -1)[:, :F].bool()


@dataclasses.dataclass
class LookaheadReport:
    layer: int                 # the predicted layer is layer + 1
    recall_standard: float     # its own predictor on its own input
    recall_lookahead: float    # the lookahead predictor on the previous layer's input
    precision_lookahead: float
    shared: float              # standard-predicted rows the lookahead one also names
    active: float              # fraction of (token, neuron) pairs that fire
    tokens_fit: int
    tokens_test: int


def _masks(desc_of, xs, p1, p2, b1, tau, F, batch=16):
    out = []
    Wd = (F + 31) // 32
    for t0 in range(0, xs.shape[0], batch):
        xb = xs[t0:t0 + batch].contiguous()
        nb = xb.shape[0]
        desc = desc_of(nb)
        ws = torch.zeros(B.pi_workspace_bytes(desc), dtype=torch.uint8, device=xs.device)
        m = torch.zeros(nb, Wd, dtype=torch.int32, device=xs.device)
        B.pi_predict(desc, xb, p1, p2, b1, tau, m, ws)
        out.append(_unpack(m, F))
    return torch.cat(out, 0)


def _active(w, xs, batch=16):
    """[T, F] bool: FC1 output non-zero, from pi_sparse_fc1 over every row."""
    F = w.F
    idx = torch.arange(F, dtype=torch.int32, device=xs.device)
    cnt = torch.tensor([F], dtype=torch.int32, device=xs.device)
    st = B.weights_struct(w)
    out = []
    for t0 in range(0, xs.shape[0], batch):
        xb = xs[t0:t0 + batch].contiguous()
        nb = xb.shape[0]
        desc = B.desc_of(w.d, F, w.r, nb, w.int4, w.gated)
        ws = torch.zeros(B.pi_workspace_bytes(desc), dtype=torch.uint8, device=xs.device)
        h = torch.empty(F * nb, dtype=torch.float32, device=xs.device)
        B.pi_sparse_fc1(desc, xb, st, idx, cnt, None, h, ws)
        out.append(h.view(F, nb).t() != 0)
    return torch.cat(out, 0)


def layer_inputs(layers, tokens, tau, eps):
    """Inputs of every layer for each token, through the library's stack call:
    list over layers of [T, d] fp16."""
    from .runtime import DecodeStack
    st = DecodeStack(layers, batch=1, tau=tau, eps=eps)
    per = [[] for _ in layers]
    for t in range(tokens.shape[0]):
        xs, _ = st.step_trace(tokens[t:t + 1])
        for l, x in enumerate(xs):
            per[l].append(x[0].clone())
    return [torch.stack(v) for v in per]


def evaluate(cfg, layer: int, n_fit: int, n_test: int, device="cuda", lam: float = 1e-3) -> LookaheadReport:
    from synth import make_layer, make_tokens
    B.lib()
    layers = [make_layer(cfg, l, device=device) for l in range(layer + 2)]
    toks = make_tokens(cfg, 0, n_fit + n_test, device=device)
    xin = layer_inputs(layers, toks, cfg.tau, cfg.rms_eps)
    x0, x1 = xin[layer], xin[layer + 1]
    M = fit_map(x0[:n_fit].T.float(), x1[:n_fit].T.float(), lam)
    nxt = layers[layer + 1]
    p1_look = (nxt.p1.double() @ M.to(nxt.p1.device)).to(torch.float16).contiguous()
    F = cfg.F
    desc_of = lambda nb: B.desc_of(nxt.d, F, nxt.r, nb, nxt.int4, nxt.gated)
    xt0, xt1 = x0[n_fit:].contiguous(), x1[n_fit:].contiguous()
    std = _masks(desc_of, xt1, nxt.p1, nxt.p2, nxt.b1, cfg.tau, F)
    look = _masks(desc_of, xt0, p1_look, nxt.p2, nxt.b1, cfg.tau, F)
    truth = _active(nxt, xt1)
    act = max(1, int(truth.sum().item()))
    return LookaheadReport(
        layer=layer,
        recall_standard=float((std & truth).sum().item()) / act,
        recall_lookahead=float((look & truth).sum().item()) / act,
        precision_lookahead=float((look & truth).sum().item()) / max(1, int(look.sum().item())),
        shared=float((look & std).sum().item()) / max(1, int(std.sum().item())),
        active=float(truth.float().mean().item()),
        tokens_fit=n_fit, tokens_test=n_test)


def main(argv=None):
    from synth import CONFIGS
    ap = argparse.ArgumentParser(description="lookahead predictor of layer l+1 from layer l's input")
    ap.add_argument("--config", default="c2")
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--fit", type=int, default=8192, help="tokens used to fit the map")
    ap.add_argument("--test", type=int, default=64, help="held-out tokens measured")
    ap.add_argument("--ridge", type=float, default=1e-3)
    args = ap.parse_args(argv)
    assert torch.cuda.is_available(), "needs a CUDA GPU"
    rep = evaluate(CONFIGS[args.config], args.layer, args.fit, args.test, lam=args.ridge)
    print(json.dumps(dataclasses.asdict(rep)), flush=True)


if __name__ == "__main__":
    main()
