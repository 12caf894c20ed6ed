"""Parity at the full workload shapes (the five configs), through the C ABI.

Full layers are generated on the GPU; the oracle recomputes sampled layers
and tokens (the whole layer output for each sampled token), fed with the
GPU's own layer input so each layer is checked on its own.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens
from tests.parity import close, mask_matches

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pi():
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    return P


def _check_layer(P, cfg, layer, batch, tokens, t0=0):
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    w = make_layer(cfg, layer, device=DEV)
    wh = oracle.host_layer(w.to("cpu"))
    st = DecodeStack([w], batch=batch, tau=cfg.tau)
    P.pi_ffn_layer  # the single-layer stack runs the same code path as pi_ffn_layer
    stats = []
    for s in range(tokens):
        x = make_tokens(cfg, t0 + s * batch, batch, device=DEV)
        y = st.step(x).clone()
        torch.cuda.synchronize()
        lay = P.pi_workspace_layout(st.desc)
        W = (w.F + 31) // 32
        mask = st.workspace[lay.mask:lay.mask + 4 * batch * W].view(torch.int32).cpu().numpy() \
            .view(np.uint32).reshape(batch, W)
        for b in range(batch):
            o = oracle.predict(x[b].cpu(), wh, cfg.tau)
            amb = mask_matches(mask[b], o, w.F, cfg.tau, f"{cfg.key} layer {layer} token {s}/{b}")
            stats.append(amb)
            close(y[b].cpu().numpy(), oracle.ffn_masked(x[b].cpu(), wh, mask[b]),
                  f"{cfg.key} layer {layer} token {s}/{b}")
    del st, w
    torch.cuda.empty_cache()
    return stats


def test_c1_full_run():
    P = _pi()
    _check_layer(P, CONFIGS["c1"], 0, 1, 64)


@pytest.mark.parametrize("layer", [0, 31])
def test_c2_layer(layer):
    P = _pi()
    _check_layer(P, CONFIGS["c2"], layer, 1, 2)


def test_c2_stack_chained_layers():
    """Four c2 layers chained through the inter-layer normalisation: each
    layer is checked against the oracle on the GPU's own input to that layer,
    and each normalisation against the oracle's on the GPU's layer output."""
    P = _pi()
    from activation_sparse_ffn_layer_gb300.runtime import DecodeStack
    from tests.parity import half_matches
    cfg = CONFIGS["c2"]
    W = (cfg.F + 31) // 32
    x = make_tokens(cfg, 0, 1, device=DEV)
    for l in range(4):
        w = make_layer(cfg, l, device=DEV)
        wh = oracle.host_layer(w.to("cpu"))
        st = DecodeStack([w], batch=1, tau=cfg.tau)
        y = st.step(x).clone()
        lay = P.pi_workspace_layout(st.layers[0].desc)
        torch.cuda.synchronize()
        mask = st.workspace[lay.mask:lay.mask + 4 * W].view(torch.int32).cpu().numpy().view(np.uint32)
        mask_matches(mask, oracle.predict(x[0].cpu(), wh, cfg.tau), cfg.F, cfg.tau, f"c2 layer {l}")
        close(y[0].cpu().numpy(), oracle.ffn_masked(x[0].cpu(), wh, mask), f"c2 layer {l}")
        xn = torch.empty_like(x)
        P.pi_rmsnorm_half(cfg.d, 1, y, cfg.rms_eps, xn)
        torch.cuda.synchronize()
        _, pre, band = oracle.rmsnorm_half(y[0].cpu().numpy().astype(np.float64), cfg.rms_eps)
        half_matches(xn[0].cpu().view(torch.int16).numpy().view(np.uint16), pre, band, f"norm {l}")
        x = xn
        del st, w


@pytest.mark.parametrize("batch", [1, 8, 32])
def test_c3_layer_batched(batch):
    P = _pi()
    _check_layer(P, CONFIGS["c3"], 6, batch, 1)        # layer 6 has rank 512


def test_c4_gated_layer():
    P = _pi()
    _check_layer(P, CONFIGS["c4"], 0, 1, 2)


@pytest.mark.parametrize("batch", [1, 4, 16])
def test_c5_int4_layer(batch):
    P = _pi()
    _check_layer(P, CONFIGS["c5"], 95, batch, 1)
