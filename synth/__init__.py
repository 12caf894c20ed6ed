"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Holds workload shapes (:mod:`synth.configs`) and the tensor generator
(:mod:`synth.generate`); none of the decode path's arithmetic lives here.
"""
from .configs import CONFIGS, Config, small  # noqa: F401
from .generate import (LayerWeights, make_layer, make_tokens, neuron_table,  # noqa: F401
                       zipf_probabilities, outlier_channels, hot_coverage, predictor_param_share)
from .attention import (ATTN_CONFIGS, AttnConfig, AttnWeights, make_attn, make_kv_cache,  # noqa: F401
                        decode_lengths, small_attn)
