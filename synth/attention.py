"""Seeded synthetic self-attention blocks and KV caches (head-sparse attention).

This module only manufactures inputs for the head-sparse attention block; it
holds none of the block's arithmetic (no projection, attention or softmax),
and both the CPU oracle and the CUDA library consume what it returns.

The pages describing PowerInfer note that in the self-attention block about
half of the heads contribute little for a given input (PowerInfer summary
(CSDN), section "Background", paragraph on activation sparsity) and that each
block has its own activity predictor (the unite.ai page, section on adaptive
sparsity predictors).  The shapes below are those of the model families the
pages run (OPT; LLaMA with grouped key/value heads); the numbers are seeded
random draws, no trained weights:

* ``Wqkv`` ``[(H + 2 KVH) dh, d]`` (query rows of head h at ``h dh``, key rows of
  KV head g at ``(H + g) dh``, value rows at ``(H + KVH + g) dh``) and
  ``Wot`` = Wo transposed ``[H dh, d]``: i.i.d. N(0, 1/d), so projections of a
  unit-RMS input have unit variance; biases N(0, bias_std^2);
* head firing probabilities ``p_h``: a Zipf law over the heads with mean
  ``head_rate`` (0.5: about half of the heads), assigned through a seeded
  permutation;
* the head predictor: a score matrix ``A`` ``[H, d]`` with i.i.d. N(0, 1/d)
  entries stands for what a trained predictor would learn; its rank-r
  truncated SVD gives ``P1`` ``[r, d]`` and ``P2`` ``[H, r]``, and the bias
  ``b_h = sigma_h Phi^-1(p_h)`` with ``sigma_h^2 = sum_j A_hj^2`` makes head h's
  score exceed 0 with probability ``p_h`` under unit Gaussian inputs;
* KV caches ``[B, KVH, smax, dh]``: positions below each sequence's length
  filled with N(0, 1) keys and values (the distribution of the projections),
  the rest zero.

Seeds: block ``l`` of config ``c`` uses ``5000 * c + l``; the caches use
``6000 * c + seed``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from .generate import _gen, _low_rank, zipf_probabilities


@dataclass(frozen=True)
class AttnConfig:
    key: str
    index: int
    name: str
    d: int
    heads: int             # query heads H
    kv_heads: int          # key/value heads KVH (H for multi-head attention)
    head_dim: int          # dh
    rank: int              # head predictor rank
    head_rate: float = 0.5
    zipf_s: float = 0.6
    bias_std: float = 0.02
    tau: float = 0.0       # head predicted active iff its score > tau
    prompt: int = 128      # cache length of the first decode token
    max_seq: int = 1024    # cache capacity per sequence


ATTN_CONFIGS = {
    "c1": AttnConfig(key="c1", index=1, name="OPT-125M-shaped attention block (d=768, 12 heads x 64)",
                     d=768, heads=12, kv_heads=12, head_dim=64, rank=8),
    "c2": AttnConfig(key="c2", index=2, name="OPT-6.7B-shaped attention block (d=4096, 32 heads x 128)",
                     d=4096, heads=32, kv_heads=32, head_dim=128, rank=32),
    "c3": AttnConfig(key="c3", index=3, name="OPT-30B-shaped attention block (d=7168, 56 heads x 128)",
                     d=7168, heads=56, kv_heads=56, head_dim=128, rank=56),
    "c4": AttnConfig(key="c4", index=4,
                     name="LLaMA-70B-shaped attention block (d=8192, 64 query heads, 8 KV heads x 128)",
                     d=8192, heads=64, kv_heads=8, head_dim=128, rank=64),
    "c5": AttnConfig(key="c5", index=5, name="OPT-175B-shaped attention block (d=12288, 96 heads x 128)",
                     d=12288, heads=96, kv_heads=96, head_dim=128, rank=64),
}


def small_attn(base: AttnConfig, *, d: int, heads: int, kv_heads: int, head_dim: int, rank: int,
               max_seq: int = 64, prompt: int = 8, key: str | None = None, **kw) -> AttnConfig:
    """A shrunken copy of an attention workload for tests."""
    f = dict(base.__dict__)
    f.update(dict(d=d, heads=heads, kv_heads=kv_heads, head_dim=head_dim, rank=rank, max_seq=max_seq,
                  prompt=prompt, key=key or f"{base.key}-small"))
    f.update(kw)
    return AttnConfig(**f)


@dataclass
class AttnWeights:
    d: int
    H: int
    KVH: int
    dh: int
    r: int
    wqkv: torch.Tensor     # fp16 [(H + 2 KVH) dh, d]
    bqkv: torch.Tensor     # fp16 [(H + 2 KVH) dh]
    wot: torch.Tensor      # fp16 [H dh, d]
    bo: torch.Tensor       # fp16 [d]
    p1: torch.Tensor       # fp16 [r, d]
    p2: torch.Tensor       # fp16 [H, r]
    bp: torch.Tensor       # fp16 [H]
    p_fire: torch.Tensor   # float64 [H] (CPU)

    def to(self, device) -> "AttnWeights":
        kw = {k: (v.to(device) if isinstance(v, torch.Tensor) and k != "p_fire" else v)
              for k, v in self.__dict__.items()}
        return AttnWeights(**kw)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for k, t in self.__dict__.items()
                   if isinstance(t, torch.Tensor) and k != "p_fire")


def make_attn(cfg: AttnConfig, layer: int = 0, device="cpu") -> AttnWeights:
    d, H, KVH, dh = cfg.d, cfg.heads, cfg.kv_heads, cfg.head_dim
    assert H % KVH == 0
    r = min(cfg.rank, H, d)
    g = _gen(5000 * cfg.index + layer, device)
    std = d ** -0.5
    rows = (H + 2 * KVH) * dh
    wqkv = (torch.randn(rows, d, generator=g, device=device) * std).to(torch.float16)
    bqkv = (torch.randn(rows, generator=g, device=device) * cfg.bias_std).to(torch.float16)
    wot = (torch.randn(H * dh, d, generator=g, device=device) * (H * dh) ** -0.5).to(torch.float16)
    bo = (torch.randn(d, generator=g, device=device) * cfg.bias_std).to(torch.float16)
    A = torch.randn(H, d, generator=g, device=device) * std
    perm = torch.randperm(H, generator=g, device=device).cpu()
    p_rank = zipf_probabilities(H, cfg.zipf_s, cfg.head_rate)
    p_fire = torch.empty(H, dtype=torch.float64)
    p_fire[perm] = p_rank
    sigma = torch.sqrt((A * A).sum(dim=1)).double().cpu()
    bp = (sigma * torch.special.ndtri(p_fire)).to(torch.float16)
    p1, p2 = _low_rank(A, r, g)
    return AttnWeights(d=d, H=H, KVH=KVH, dh=dh, r=r, wqkv=wqkv.contiguous(), bqkv=bqkv.contiguous(),
                       wot=wot.contiguous(), bo=bo.contiguous(), p1=p1.to(torch.float16).contiguous(),
                       p2=p2.to(torch.float16).contiguous(), bp=bp.to(device).contiguous(), p_fire=p_fire)


def make_kv_cache(cfg: AttnConfig, lengths, seed: int = 0, device="cpu", max_seq: int | None = None):
    """Key and value caches [B, KVH, smax, dh] fp16 for sequences whose first
    ``lengths[b]`` positions are filled (N(0, 1)), the rest zero."""
    smax = cfg.max_seq if max_seq is None else max_seq
    B = len(lengths)
    g = _gen(6000 * cfg.index + seed, device)
    k = torch.randn(B, cfg.kv_heads, smax, cfg.head_dim, generator=g, device=device)
    v = torch.randn(B, cfg.kv_heads, smax, cfg.head_dim, generator=g, device=device)
    pos = torch.arange(smax, device=device)
    for b, n in enumerate(lengths):
        assert 0 <= n < smax
        k[b, :, pos >= n] = 0
        v[b, :, pos >= n] = 0
    return k.to(torch.float16).contiguous(), v.to(torch.float16).contiguous()


def decode_lengths(cfg: AttnConfig, batch: int, step: int = 0):
    """Cache lengths of a batch at decode step ``step``: the prompt plus the
    step, ragged across sequences by a fixed offset pattern (below max_seq)."""
    out = []
    for b in range(batch):
        n = cfg.prompt + step + (37 * b) % max(1, cfg.max_seq // 8)
        out.append(min(n, cfg.max_seq - 1))
    return out
