"""pi_sparse_fc2_noalloc: FC2 for callers that cannot allocate device memory
(for example a plug-in whose host framework owns the whole device memory pool
and offers it no allocation hook).  It must give exactly the result of
pi_sparse_fc2 with a caller workspace, on two calls in a row with different
inputs, on every FC2 path the plan can take, and match the oracle's FC2 on
the same h and index list.

Kept in a file of its own that pytest collects last; it builds and loads the
library itself, so it also runs alone in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(P, cfg, batch, token0):
    """One layer's FC2 inputs (h, idx, count from the library's own predictor,
    compaction and FC1) and pi_sparse_fc2's output with a workspace filled
    with NaN bytes, so a partial-sum slot that the reduction reads without the
    same call having written it would show up."""
    w = make_layer(cfg, 0, device=DEV)
    x = make_tokens(cfg, token0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    nbytes = P.pi_workspace_bytes(desc)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    mask = torch.zeros(batch, (w.F + 31) // 32, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    h = torch.zeros(w.F * batch, dtype=torch.float32, device=DEV)
    wsx = P.weights_struct(w)
    P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask if batch > 1 else None, h, ws)
    ws_nan = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    y_ref = torch.empty(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc2(desc, h, idx, cnt, wsx, y_ref, ws_nan)
    return w, desc, wsx, h, idx, cnt, y_ref


@pytest.mark.parametrize("kind,cfg,batch", [
    # per-token CUDA-core kernels with a split reduction
    ("fp16-b1", small(CONFIGS["c2"], d=1024, F=4096, rank=64), 1),
    # streamed CUDA-core path (2..8 tokens)
    ("fp16-b4", small(CONFIGS["c3"], d=1024, F=4096, rank=64), 4),
    # tensor-core path (16..32 tokens)
    ("fp16-b16", small(CONFIGS["c3"], d=1024, F=4096, rank=64), 16),
    # gated, LLaMA-width rows, 32 tokens: FC1's split partials exceed the
    # array, FC2's own fit, so the call must be accepted
    ("gated-b32", small(CONFIGS["c4"], d=8192, F=2048, rank=64), 32),
    # INT4 streamed CUDA-core path
    ("int4-b3", small(CONFIGS["c5"], d=1024, F=4100, rank=64), 3),
    # INT4 tensor-core FC2 (16 tokens)
    ("int4-b16", small(CONFIGS["c5"], d=1024, F=4100, rank=64), 16),
])
def test_noalloc_fc2_matches_workspace_fc2_twice(kind, cfg, batch):
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    cases = [_case(P, cfg, batch, 0), _case(P, cfg, batch, 17)]     # two different inputs
    outs = []
    for w, desc, wsx, h, idx, cnt, y_ref in cases:                  # two calls in a row
        y = torch.full_like(y_ref, float("nan"))
        P.pi_sparse_fc2_noalloc(desc, h, idx, cnt, wsx, y)
        outs.append(y)
    torch.cuda.synchronize()
    for n, ((w, desc, wsx, h, idx, cnt, y_ref), y) in enumerate(zip(cases, outs)):
        # same kernels and the same fixed reduction order: identical bits
        assert torch.equal(y, y_ref), f"{kind} call {n}: differs from pi_sparse_fc2"
        c = int(cnt.item())
        ix = idx[:c].cpu().numpy()
        hh = h[:c * batch].cpu().numpy().astype(np.float64).reshape(c, batch)
        wh = oracle.host_layer(w.to("cpu"))
        for b in range(batch):
            yo = oracle.fc2(hh[:, b], wh, ix)
            close(y[b].cpu().numpy(), yo, f"{kind} call {n} token {b} vs oracle")
    assert not torch.equal(cases[0][6], cases[1][6])


def test_noalloc_fc2_rejects_too_large():
    """A descriptor whose FC2 partial sums alone exceed the 8 MiB array is
    refused before anything is launched.  d = 65536 at 32 tokens: the
    tensor-core FC2 needs at least (d/128 + 2) tiles x 32 x 128 floats on any
    SM count, above 2 Mi floats.  The buffers are still sized for the
    descriptor, so a wrongly accepted call could not write out of bounds."""
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    d, F, B = 65536, 64, 32
    desc = P.desc_of(d, F, 64, B)
    h = torch.zeros(F * B, dtype=torch.float32, device=DEV)
    idx = torch.zeros(F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = torch.zeros(B, d, dtype=torch.float32, device=DEV)
    w2t = torch.zeros(F, d, dtype=torch.float16, device=DEV)
    b2 = torch.zeros(d, dtype=torch.float16, device=DEV)
    s = P.binding.pi_layer_weights()
    s.w2t = P.binding._ptr(w2t)
    s.b2 = P.binding._ptr(b2)
    with pytest.raises(P.PiError) as e:
        P.pi_sparse_fc2_noalloc(desc, h, idx, cnt, s, y)
    assert e.value.status == 5
