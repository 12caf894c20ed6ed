"""pi_sparse_fc2_noalloc (FC2 for callers that cannot allocate device memory,
e.g. a plug-in whose host framework owns the device memory pool) gives the
same result as pi_sparse_fc2 with a caller workspace, on two calls in a row.

Kept in a file of its own that pytest collects last; it builds and loads the
library itself, so it also runs alone in a fresh process."""
import numpy as np
import pytest
import torch

from synth import CONFIGS, make_layer, make_tokens, small
from tests.parity import close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(P, cfg, batch, token0):
    w = make_layer(cfg, 0, device=DEV)
    x = make_tokens(cfg, token0, batch, device=DEV)
    desc = P.layer_desc(w, batch)
    ws = torch.zeros(P.pi_workspace_bytes(desc), dtype=torch.uint8, device=DEV)
    mask = torch.zeros(batch, (w.F + 31) // 32, dtype=torch.int32, device=DEV)
    P.pi_predict(desc, x, w.p1, w.p2, w.b1, cfg.tau, mask, ws)
    idx = torch.zeros(w.F, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int32, device=DEV)
    P.pi_compact(desc, mask, None, idx, None, cnt)
    h = torch.zeros(w.F * batch, dtype=torch.float32, device=DEV)
    wsx = P.weights_struct(w)
    P.pi_sparse_fc1(desc, x, wsx, idx, cnt, mask if batch > 1 else None, h, ws)
    y_ref = torch.empty(batch, w.d, dtype=torch.float32, device=DEV)
    P.pi_sparse_fc2(desc, h, idx, cnt, wsx, y_ref, ws)
    return w, desc, wsx, h, idx, cnt, y_ref


@pytest.mark.parametrize("kind,cfg,batch", [
    ("fp16", small(CONFIGS["c2"], d=1024, F=4096, rank=64), 1),
    ("int4", small(CONFIGS["c5"], d=1024, F=4100, rank=64), 3),
])
def test_noalloc_fc2_matches_workspace_fc2_twice(kind, cfg, batch):
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    cases = [_case(P, cfg, batch, 0), _case(P, cfg, batch, 17)]     # two different inputs
    outs = []
    for w, desc, wsx, h, idx, cnt, y_ref in cases:                  # two calls in a row
        y = torch.full_like(y_ref, float("nan"))
        P.pi_sparse_fc2_noalloc(desc, h, idx, cnt, wsx, y)
        outs.append((y, y_ref))
    torch.cuda.synchronize()
    for n, (y, y_ref) in enumerate(outs):
        close(y.cpu().numpy(), y_ref.cpu().numpy(), f"{kind} call {n}")
    assert not torch.equal(outs[0][1], outs[1][1])


def test_noalloc_fc2_rejects_too_large():
    import activation_sparse_ffn_layer_gb300 as P
    P.lib()
    desc = P.desc_of(16384, 65536, 64, 32)      # partial sums far beyond the 8 MiB array
    z = torch.zeros(16, dtype=torch.float32, device=DEV)
    zi = torch.zeros(16, dtype=torch.int32, device=DEV)
    s = P.binding.pi_layer_weights()
    s.w2t = P.binding._ptr(torch.zeros(8, dtype=torch.float16, device=DEV))
    s.b2 = s.w2t
    with pytest.raises(P.PiError) as e:
        P.pi_sparse_fc2_noalloc(desc, z, zi, zi, s, z)
    assert e.value.status == 5
