"""The five synthetic decode workloads (shapes, sparsity and run lengths).

Each workload is a ReLU FFN layer, or a stack of them, shaped like a published
model and filled with seeded random numbers: no trained weights, predictors or
prompt datasets are used.  The firing statistics follow the power-law locality
described in the PowerInfer summary (CSDN), section "Introduction" (a small hot
set of neurons carries most activations; the rest depend on the input), and the
model families are the ones named in its section "Implementation" (OPT, LLaMA).

Every number the method's arithmetic depends on is a field here; the generator
in :mod:`synth.generate` turns a config into tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Config:
    key: str                 # "c1" .. "c5"
    index: int               # 1 .. 5, used in the seeds
    name: str                # what the workload is, with its shape
    layers: int
    d: int                   # model width
    F: int                   # FFN width (neurons)
    rank: int                # predictor rank (per-layer override: rank_rule)
    zipf_s: float            # Zipf exponent of the firing probabilities
    mean_rate: float         # mean firing probability per layer
    tokens: int              # decode steps of the run
    batches: tuple = (1,)
    gated: bool = False      # LLaMA-style gate/up projection with ReLU on the gate
    int4: bool = False       # W1/W2 in symmetric INT4, group 32 along d, fp16 scales
    outliers: int = 0        # input channels scaled by outlier_scale (layer-0 input)
    outlier_scale: float = 8.0
    weight_std: float = 0.02
    tau: float = -0.05       # predictor threshold: neuron predicted active iff score > tau
    hot_frac: float = 0.2    # fraction of neurons packed first in the neuron table
    per_layer_rates: tuple = ()   # (lo, hi) of linearly spaced per-layer rates, else ()
    has_b2: bool = True
    rms_eps: float = 1e-6

    # ---- derived -------------------------------------------------------
    def layer_rate(self, layer: int) -> float:
        """Mean firing probability of one layer."""
        if not self.per_layer_rates:
            return self.mean_rate
        return _layer_rates(self)[layer]

    def layer_rank(self, layer: int) -> int:
        """Predictor rank of one layer.

        With per-layer rates the rank grows linearly with the layer's firing
        rate from 64 (sparsest) to 512 (densest), rounded to a multiple of 32:
        a sparser layer gets a smaller predictor (PowerInfer summary (CSDN),
        section "Adaptive sparse predictor": layers with higher sparsity make
        the active set easier to find and allow a smaller predictor).
        """
        if not self.per_layer_rates:
            return self.rank
        lo, hi = self.per_layer_rates
        m = _layer_rates(self)[layer]
        r = 64 + 448 * (m - lo) / (hi - lo)
        return int(32 * round(r / 32))

    def max_rank(self) -> int:
        return max(self.layer_rank(l) for l in range(self.layers))

    def n_hot(self) -> int:
        return int(math.ceil(self.hot_frac * self.F))


def _layer_rates(cfg: Config) -> list:
    """Per-layer mean rates: linearly spaced over (lo, hi), assigned to the
    layers by a seeded permutation (a pure function of the config index)."""
    import random
    lo, hi = cfg.per_layer_rates
    L = cfg.layers
    rates = [lo + (hi - lo) * i / (L - 1) for i in range(L)] if L > 1 else [0.5 * (lo + hi)]
    rng = random.Random(7919 * cfg.index)
    rng.shuffle(rates)
    return rates


CONFIGS = {
    "c1": Config(key="c1", index=1, name="OPT-125M-shaped ReLU FFN layer (d=768, F=3072, r=64)",
                 layers=1, d=768, F=3072, rank=64, zipf_s=1.1, mean_rate=0.10,
                 tokens=64, outliers=2),
    "c2": Config(key="c2", index=2, name="OPT-6.7B-shaped FFN stack (32 x d=4096, F=16384, r=256)",
                 layers=32, d=4096, F=16384, rank=256, zipf_s=1.1, mean_rate=0.10,
                 tokens=128),
    "c3": Config(key="c3", index=3, name="OPT-30B-shaped FFN stack (48 x d=7168, F=28672, r=64..512)",
                 layers=48, d=7168, F=28672, rank=288, zipf_s=1.2, mean_rate=0.08,
                 tokens=64, batches=(1, 2, 4, 8, 16, 32), per_layer_rates=(0.04, 0.12)),
    "c4": Config(key="c4", index=4, name="LLaMA-70B-shaped ReLU-gated FFN stack (80 x d=8192, F=28672, r=512)",
                 layers=80, d=8192, F=28672, rank=512, zipf_s=1.0, mean_rate=0.12,
                 tokens=64, gated=True, has_b2=False),
    "c5": Config(key="c5", index=5, name="OPT-175B-shaped INT4 FFN stack (96 x d=12288, F=49152, r=1024)",
                 layers=96, d=12288, F=49152, rank=1024, zipf_s=1.1, mean_rate=0.06,
                 tokens=64, batches=(1, 4, 16), int4=True),
}


def small(base: Config, *, d: int, F: int, rank: int, layers: int = 1, tokens: int = 4,
          key: str | None = None, **kw) -> Config:
    """A shrunken copy of a workload for tests: same statistics, smaller shape."""
    fields = dict(base.__dict__)
    fields.update(dict(d=d, F=F, rank=rank, layers=layers, tokens=tokens,
                       key=key or f"{base.key}-small"))
    fields.update(kw)
    if fields["per_layer_rates"] and layers == 1:
        fields["per_layer_rates"] = ()
    return Config(**fields)
