"""Seeded synthetic layers and decode tokens for the sparse-FFN workloads.

This module only manufactures inputs.  It holds none of the decode path's
arithmetic (no predictor, compaction, FFN, dequantisation or normalisation);
both the CPU oracle and the CUDA library consume the tensors it returns.

What it builds, per layer (all per-neuron arrays in *storage order*, i.e. the
order of the neuron table, hot neurons first):

* ``W1`` (or the gate ``Wg``), ``W2^T`` and, for gated layers, ``Wu``: i.i.d.
  N(0, weight_std^2), drawn in original neuron order;
* firing probabilities ``p_i``: a Zipf(s) law over the ranks, capped at 0.999
  and scaled by bisection so that their mean is the configured rate, assigned
  to neurons through a seeded permutation (the power-law locality of the
  PowerInfer summary (CSDN), section "Introduction");
* ``b1_i = sigma_i * Phi^-1(p_i)`` with ``sigma_i^2 = sum_j W1_ij^2 var(x_j)``, so
  that neuron ``i`` fires (``W1_i.x + b1_i > 0``) with probability ``p_i`` under
  Gaussian inputs;
* the neuron table (PowerInfer summary (CSDN), section "Neuron placement and
  management": a table maps each stored neuron to its original position): the
  ``ceil(hot_frac * F)`` most probable neurons first, by descending ``p``, then
  the rest in original order;
* the predictor: the rank-r truncated SVD ``W1 ~= U S V^T`` gives ``P1 = V_r^T``
  ``[r, d]`` and ``P2 = U_r S_r`` ``[F, r]`` (the predictor bias is ``b1``).  The
  pages train small MLP predictors offline (section "Adaptive sparse
  predictor"); with no training data a low-rank linear map of the layer's own
  weights stands in;
* INT4 layers: symmetric group-32 quantisation along ``d`` with fp16 scales
  ``s = fp16(absmax / 7)``, ``q = clamp(rint(w / s), -8, 7)``, two codes per byte
  (low nibble = even element).  Calibration and the SVD use ``q * s``.

Seeds: layer ``l`` of config ``c`` uses ``1000 * c + l``; token ``t`` uses
``2000 * c + t``; the outlier channels use ``1000 * c + 999``.  Random streams
depend on the device the tensors are drawn on; a comparison always feeds the
same drawn tensors to both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, fields
from typing import Optional

import torch

from .configs import Config


@dataclass
class LayerWeights:
    d: int
    F: int
    r: int
    gated: bool
    int4: bool
    b1: torch.Tensor                   # fp16 [F]      FC1 (gate) bias, also the predictor bias
    b2: torch.Tensor                   # fp16 [d]
    p1: torch.Tensor                   # fp16 [r, d]
    p2: torch.Tensor                   # fp16 [F, r]
    table: torch.Tensor                # int32 [F]     storage row -> original neuron id
    p_fire: torch.Tensor               # float64 [F]   firing probability, original order (CPU)
    w1: Optional[torch.Tensor] = None  # fp16 [F, d]   FC1 (gate) rows
    wu: Optional[torch.Tensor] = None  # fp16 [F, d]   up-projection rows (gated)
    w2t: Optional[torch.Tensor] = None  # fp16 [F, d]  FC2 columns stored as rows
    w1_q: Optional[torch.Tensor] = None  # uint8 [F, d/2]
    w1_s: Optional[torch.Tensor] = None  # fp16 [F, d/32]
    w2t_q: Optional[torch.Tensor] = None
    w2t_s: Optional[torch.Tensor] = None
    w1_recon: Optional[torch.Tensor] = None  # fp32 [F, d] q*s of the INT4 FC1 rows (keep_recon only)

    def tensors(self):
        return {f.name: getattr(self, f.name) for f in fields(self)
                if isinstance(getattr(self, f.name), torch.Tensor)}

    def to(self, device) -> "LayerWeights":
        kw = {}
        for f in fields(self):
            v = getattr(self, f.name)
            if isinstance(v, torch.Tensor) and f.name != "p_fire":
                v = v.to(device)
            kw[f.name] = v
        return LayerWeights(**kw)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for k, t in self.tensors().items()
                   if k not in ("p_fire", "w1_recon"))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def outlier_channels(cfg: Config) -> list:
    """The input channels scaled by ``outlier_scale`` (fixed for a run)."""
    if cfg.outliers == 0:
        return []
    g = _gen(1000 * cfg.index + 999, "cpu")
    return sorted(torch.randperm(cfg.d, generator=g)[: cfg.outliers].tolist())


def zipf_probabilities(F: int, s: float, mean: float, cap: float = 0.999) -> torch.Tensor:
    """Firing probability by rank (rank 1 first): ``min(c * rank^-s, cap)`` with
    ``c`` found by bisection so that the mean is ``mean``.  float64, CPU."""
    rank = torch.arange(1, F + 1, dtype=torch.float64)
    raw = rank.pow(-s)
    lo, hi = 0.0, 1.0
    while torch.clamp(hi * raw, max=cap).mean().item() < mean:
        hi *= 2.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if torch.clamp(mid * raw, max=cap).mean().item() < mean:
            lo = mid
        else:
            hi = mid
    return torch.clamp(hi * raw, max=cap)


def _orth(Y: torch.Tensor) -> torch.Tensor:
    """Orthonormal basis of the columns of Y (Cholesky-QR through an fp64
    eigendecomposition of the small Gram matrix, done on the CPU)."""
    G = (Y.T @ Y).double().cpu()
    evals, evecs = torch.linalg.eigh(G)
    evals = torch.clamp(evals, min=float(evals.max()) * 1e-13)
    return Y @ (evecs / torch.sqrt(evals)).to(Y.device, Y.dtype)


def _low_rank(W: torch.Tensor, r: int, g: torch.Generator, oversample: int = 16, power_iters: int = 2):
    """Rank-r truncated SVD factors (P1 = V_r^T, P2 = U_r S_r) of an fp32 matrix.

    Exact SVD (fp64, CPU) for small matrices; otherwise the randomized range
    finder with power iterations of Halko, Martinsson and Tropp (SIAM Review
    2011): large products on W's device, small factorisations in fp64 on the CPU.
    """
    F, d = W.shape
    r = min(r, F, d)
    if F * d <= 4_000_000:
        U, S, Vh = torch.linalg.svd(W.double().cpu(), full_matrices=False)
        return Vh[:r].float().to(W.device), (U[:, :r] * S[:r]).float().to(W.device)
    k = min(r + oversample, d)
    omega = torch.randn(d, k, generator=g, device=W.device, dtype=torch.float32)
    Q = _orth(W @ omega)
    for _ in range(power_iters):
        Z = _orth(W.T @ Q)
        Q = _orth(W @ Z)
    Bm = Q.T @ W                                   # [k, d]
    evals, evecs = torch.linalg.eigh((Bm @ Bm.T).double().cpu())   # Bm Bm^T = Ub S^2 Ub^T
    order = torch.argsort(evals, descending=True)[:r]
    S = torch.sqrt(torch.clamp(evals[order], min=0.0))
    Ub = evecs[:, order]
    Ub_d = Ub.to(W.device, torch.float32)
    S_d = S.to(W.device, torch.float32)
    Vh = (Ub_d.T @ Bm) / torch.clamp(S_d, min=1e-30)[:, None]      # S^-1 Ub^T Bm
    U = Q @ Ub_d
    return Vh.contiguous(), (U * S_d).contiguous()


def _quantize_g32(w: torch.Tensor):
    """Symmetric INT4, groups of 32 along the row: returns (packed uint8 [F, d/2],
    scales fp16 [F, d/32], reconstruction q*s as fp32)."""
    F, d = w.shape
    grp = w.reshape(F, d // 32, 32)
    s16 = (grp.abs().amax(dim=2) / 7.0).to(torch.float16)
    s = s16.float().unsqueeze(2)
    safe = torch.where(s == 0, torch.ones_like(s), s)
    q = torch.clamp(torch.round(grp / safe), -8, 7)       # torch.round: half to even
    q = torch.where(s == 0, torch.zeros_like(q), q)
    recon = (q * s).reshape(F, d)
    qi = q.to(torch.int16).reshape(F, d)
    lo = (qi[:, 0::2] & 0xF)
    hi = (qi[:, 1::2] & 0xF)
    packed = (lo | (hi << 4)).to(torch.uint8)
    return packed.contiguous(), s16.contiguous(), recon


def neuron_table(p_fire: torch.Tensor, n_hot: int) -> torch.Tensor:
    """Storage row -> original id: hot neurons by descending p (ties by id),
    then the cold ones in original order."""
    order = torch.argsort(-p_fire, stable=True)
    hot = order[:n_hot]
    is_hot = torch.zeros(p_fire.numel(), dtype=torch.bool)
    is_hot[hot] = True
    cold = torch.nonzero(~is_hot).flatten()
    return torch.cat([hot, cold]).to(torch.int32)


def make_layer(cfg: Config, layer: int, device="cpu", *, table_override: Optional[torch.Tensor] = None,
               keep_recon: bool = False) -> LayerWeights:
    """Draw one layer of a workload.  ``table_override`` (a permutation of
    ``range(F)``) replaces the hot-first neuron table; the layer is otherwise
    identical, which lets tests check that the table order does not matter.
    ``keep_recon`` keeps, for INT4 layers, the fp32 reconstruction of the FC1
    rows that the calibration and the factorisation used (storage order)."""
    d, F = cfg.d, cfg.F
    r = min(cfg.layer_rank(layer), d, F)
    g = _gen(1000 * cfg.index + layer, device)
    std = cfg.weight_std
    w1 = torch.randn(F, d, generator=g, device=device) * std
    w2t = torch.randn(F, d, generator=g, device=device) * std
    wu = torch.randn(F, d, generator=g, device=device) * std if cfg.gated else None
    b2 = (torch.randn(d, generator=g, device=device) * std) if cfg.has_b2 else torch.zeros(d, device=device)
    perm = torch.randperm(F, generator=g, device=device).cpu()

    out = {}
    if cfg.int4:
        w1_q, w1_s, w1 = _quantize_g32(w1)          # w1 becomes the reconstruction q*s
        w2t_q, w2t_s, _ = _quantize_g32(w2t)
        out.update(w1_q=w1_q, w1_s=w1_s, w2t_q=w2t_q, w2t_s=w2t_s)
    else:
        w1 = w1.to(torch.float16).float()           # calibrate on the stored fp16 values
        out["w2t"] = w2t.to(torch.float16)
        if cfg.gated:
            out["wu"] = wu.to(torch.float16)

    # firing probabilities and calibrated bias
    p_rank = zipf_probabilities(F, cfg.zipf_s, cfg.layer_rate(layer))
    p_fire = torch.empty(F, dtype=torch.float64)
    p_fire[perm] = p_rank
    var = torch.ones(d, device=device)
    for ch in outlier_channels(cfg):
        var[ch] = cfg.outlier_scale ** 2
    sigma = torch.sqrt((w1 * w1) @ var).double().cpu()
    b1 = (sigma * torch.special.ndtri(p_fire)).to(torch.float16)

    p1, p2 = _low_rank(w1, r, g)

    table = neuron_table(p_fire, cfg.n_hot()) if table_override is None else table_override.to(torch.int32).cpu()
    rows = table.long().to(device)
    if not cfg.int4:
        out["w1"] = w1.to(torch.float16)[rows].contiguous()
        out["w2t"] = out["w2t"][rows].contiguous()
        if cfg.gated:
            out["wu"] = out["wu"][rows].contiguous()
    else:
        for k in ("w1_q", "w1_s", "w2t_q", "w2t_s"):
            out[k] = out[k][rows].contiguous()
        if keep_recon:
            out["w1_recon"] = w1[rows].contiguous()
    return LayerWeights(
        d=d, F=F, r=r, gated=cfg.gated, int4=cfg.int4,
        b1=b1.to(device)[rows].contiguous(),
        b2=b2.to(torch.float16).contiguous(),
        p1=p1.to(torch.float16).contiguous(),
        p2=p2.to(torch.float16)[rows].contiguous(),
        table=table.to(device),
        p_fire=p_fire,
        **out,
    )


def make_tokens(cfg: Config, t0: int, count: int, device="cpu") -> torch.Tensor:
    """Layer-0 inputs of tokens ``t0 .. t0+count-1``: N(0, 1) per channel, the
    outlier channels scaled, rounded to fp16.  Shape [count, d]."""
    chans = outlier_channels(cfg)
    xs = []
    for t in range(t0, t0 + count):
        g = _gen(2000 * cfg.index + t, device)
        x = torch.randn(cfg.d, generator=g, device=device)
        for ch in chans:
            x[ch] *= cfg.outlier_scale
        xs.append(x)
    return torch.stack(xs).to(torch.float16).contiguous()


def hot_coverage(w: LayerWeights, n_hot: int) -> float:
    """Share of the expected activations carried by the hot prefix of the table."""
    p = w.p_fire
    hot = w.table[:n_hot].long().cpu()
    return float(p[hot].sum() / p.sum())


def predictor_param_share(cfg: Config) -> float:
    """Predictor parameters over FFN parameters, summed over the stack."""
    m = 3 if cfg.gated else 2
    pred = sum(cfg.layer_rank(l) * (cfg.d + cfg.F) for l in range(cfg.layers))
    return pred / (cfg.layers * m * cfg.d * cfg.F)
