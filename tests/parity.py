"""Shared helpers of the parity tests: tolerances and the mask rule.

Floating outputs must meet max-abs error <= 2e-3 and relative L2 error <= 1e-3
against the fp64 oracle (fp16 weights, fp32 accumulation).  Masks and index
lists must be bit-exact, except that a predictor score lying within the
oracle's guard band of the threshold may fall on either side (several answers
are correct there; fp32 rounding in any summation order can move it).
"""
import numpy as np

MAX_ABS = 2e-3
REL_L2 = 1e-3


def close(gpu, ref, what="", max_abs=MAX_ABS, rel_l2=REL_L2):
    g = np.asarray(gpu, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - r)
    ma = float(err.max()) if err.size else 0.0
    nr = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / nr) if nr > 0 else 0.0
    assert ma <= max_abs, f"{what}: max-abs {ma:.3e} > {max_abs}"
    assert rel <= rel_l2 or nr == 0, f"{what}: rel-L2 {rel:.3e} > {rel_l2}"
    return ma, rel


def unpack_mask(words, F):
    w = np.asarray(words, dtype=np.uint32).ravel()
    bits = ((w[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).ravel()
    return bits[:F]


def mask_matches(gpu_words, oracle_out, F, tau, what=""):
    """GPU mask vs oracle: identical outside the guard band; returns how many
    in-band bits differ.  Bits past F must be 0."""
    gw = np.asarray(gpu_words, dtype=np.uint32).ravel()
    gb = unpack_mask(gw, F)
    ob = unpack_mask(oracle_out["mask"], F)
    tail = ((gw[:, None] >> np.arange(32, dtype=np.uint32)[None, :]) & 1).astype(bool).ravel()[F:]
    assert not tail.any(), f"{what}: mask bits set past F"
    amb = np.abs(oracle_out["s"] - np.float64(np.float32(tau))) <= oracle_out["band"]
    bad = (gb != ob) & ~amb
    assert not bad.any(), f"{what}: {int(bad.sum())} mask bits differ outside the guard band " \
                          f"(first at {int(np.nonzero(bad)[0][0])})"
    return int(((gb != ob) & amb).sum())


def half_matches(gpu_bits, pre, band, what=""):
    """fp16 outputs vs the oracle's pre-rounding values: equal to the rounding
    of some value within [pre - band, pre + band]."""
    import oracle
    g = np.asarray(gpu_bits, dtype=np.uint16).ravel().view(np.float16).astype(np.float64)
    lo = oracle.double_to_half(pre - band).view(np.float16).astype(np.float64)
    hi = oracle.double_to_half(pre + band).view(np.float16).astype(np.float64)
    bad = (g < lo) | (g > hi)
    assert not bad.any(), f"{what}: {int(bad.sum())} fp16 outputs outside the rounding band"
