"""The batch-1 persistent kernel's plan, checked on the host for a 152-SM
device (pi_stack_plan_for queries no GPU): which predictor mode each workload
shape takes (slices staged whole in shared memory, or P2 streamed through the
ring of 16-row slots), the ring and FC-row slot counts, the shared-memory
budget, and the shapes the persistent kernel leaves to the per-step kernels."""
import ctypes as C

import numpy as np
import pytest

from synth import CONFIGS

SMS = 152
SMEM_MAX = 227 * 1024          # dynamic shared memory a block may use on sm_103a
KIB = 1024


@pytest.fixture(scope="module")
def P():
    import __graft_entry__
    __graft_entry__.build()
    import activation_sparse_ffn_layer_gb300 as P
    return P


def _plan(P, d, F, r, L=2, int4=False, gated=False, batch=1, ranks=None, sms=SMS):
    desc = P.desc_of(d, F, r, batch, int4, gated)
    arr = None if ranks is None else (C.c_int * len(ranks))(*ranks)
    return P.pi_stack_plan_for(desc, L, sms, arr)


def _cfg_plan(P, key):
    cfg = CONFIGS[key]
    ranks = [cfg.layer_rank(l) for l in range(cfg.layers)]
    return _plan(P, cfg.d, cfg.F, max(ranks), L=cfg.layers, int4=cfg.int4, gated=cfg.gated, ranks=ranks)


def _check_invariants(p, gated):
    assert p.fused == 1 and p.ctas == SMS
    assert 0 < p.smem_bytes <= SMEM_MAX
    if p.pred_in_smem:
        assert p.p2_ring_slots == 0
    else:
        assert 2 <= p.p2_ring_slots <= 8
    assert (4 if gated else 2) <= p.fc_row_slots <= 32


def test_workload_shapes_take_the_expected_modes(P):
    # OPT-175B-shaped INT4 stack: P2 (100 MB per layer) streams through six 32 KB slots
    c5 = _cfg_plan(P, "c5")
    _check_invariants(c5, False)
    assert c5.pred_in_smem == 0 and c5.p2_ring_slots == 6
    # LLaMA-70B-shaped gated stack: eight 16 KB slots
    c4 = _cfg_plan(P, "c4")
    _check_invariants(c4, True)
    assert c4.pred_in_smem == 0 and c4.p2_ring_slots == 8
    # OPT-30B-shaped stack: its largest ranks (512) need the ring
    c3 = _cfg_plan(P, "c3")
    _check_invariants(c3, False)
    assert c3.pred_in_smem == 0
    # OPT-6.7B- and OPT-125M-shaped stacks: a block's predictor share fits whole
    for key in ("c2", "c1"):
        p = _cfg_plan(P, key)
        _check_invariants(p, False)
        assert p.pred_in_smem == 1, key


def test_the_shared_memory_budget_holds_over_many_shapes(P):
    rng = np.random.default_rng(7)
    seen = {"smem": 0, "ring": 0, "per-step": 0}
    for _ in range(300):
        int4 = bool(rng.integers(2))
        gated = not int4 and bool(rng.integers(2))
        d = int(rng.integers(1, 49)) * 256
        F = int(rng.integers(64, 60000))
        r = int(rng.integers(1, min(d, 2048) // 8 + 1)) * 8
        L = int(rng.integers(1, 97))
        p = _plan(P, d, F, r, L=L, int4=int4, gated=gated)
        if p.fused:
            _check_invariants(p, gated)
            seen["smem" if p.pred_in_smem else "ring"] += 1
        else:
            seen["per-step"] += 1
            assert p.ctas == 0 and p.smem_bytes == 0
    assert all(v > 0 for v in seen.values()), seen


def test_shapes_left_to_the_per_step_kernels(P):
    # a 16-row P2 unit of rank 4096 is 128 KB: fewer than two ring slots fit
    assert _plan(P, 4096, 5000, 4096).fused == 0
    # more than one token per step
    assert _plan(P, 4096, 16384, 256, batch=4).fused == 0
    # and the same shape at batch 1 does run persistently
    assert _plan(P, 4096, 16384, 256).fused == 1


def test_plan_depends_on_the_sm_count_not_on_a_device(P):
    a = _plan(P, 12288, 49152, 1024, int4=True, sms=152)
    b = _plan(P, 12288, 49152, 1024, int4=True, sms=148)
    assert a.ctas == 152 and b.ctas == 148
    # fewer blocks own more 16-row units each; both still stream P2 through the ring
    assert a.pred_in_smem == b.pred_in_smem == 0


def test_bad_sm_count_is_rejected(P):
    desc = P.desc_of(1024, 4096, 64)
    for sms in (0, -1, 5000):
        with pytest.raises(P.PiError):
            P.pi_stack_plan_for(desc, 1, sms)
