"""Pins of the oracle's number handling: binary16 decode/encode and INT4 codes.

Each check compares against something other than the oracle: the IEEE 754
binary16 definition (hand-worked fixtures), numpy's float16 conversion (a
library routine), or hand-decoded INT4 rows.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def test_half_decode_fixture():
    for val, bits in _rows("half_bits.txt"):
        got = oracle.half_to_double(np.array([int(bits, 16)], np.uint16))[0]
        assert got == float(val) and np.signbit(got) == np.signbit(float(val)), (val, bits, got)


def test_half_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_half_encode_fixture():
    for val, bits in ((r[0], r[1]) for r in _rows("half_rounding.txt")):
        got = int(oracle.double_to_half([float(val)])[0])
        assert got == int(bits, 16), (val, hex(got), bits)


def test_half_encode_matches_numpy_rounding():
    rng = np.random.default_rng(0)
    with np.errstate(invalid="ignore", over="ignore"):
        _run_encode_vs_numpy(rng)


def _run_encode_vs_numpy(rng):
    vals = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        # exact ties: midpoints of consecutive binary16 values
        (np.arange(0, 65535, 7, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
         + np.arange(1, 65536, 7, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)) / 2,
        np.array([0.0, -0.0, 65504.0, 65519.999, 65520.0, 1e9, -1e9, 2.0 ** -25, 2.0 ** -26]),
    ])
    vals = vals[np.isfinite(vals)]
    ours = oracle.double_to_half(vals)
    ref = vals.astype(np.float16).view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(vals[i], hex(ours[i]), hex(ref[i])) for i in bad[:5]]


def test_int4_rows_fixture():
    rows = {r[0]: r[1:] for r in _rows("int4_rows.txt")}
    q = np.array([int(b, 16) for b in rows["bytes"]], np.uint8).reshape(1, 32)
    s = np.array([int(b, 16) for b in rows["scales"]], np.uint16).reshape(1, 2)
    m = oracle.Matrix(q=q, scales=s)
    got = oracle.decode_row(m, 64, 0)
    want = np.array([float(v) for v in rows["group0"] + rows["group1"]])
    assert np.array_equal(got, want)


def test_int4_decode_roundtrip_of_exact_codes():
    # a row whose values are exactly k * s for codes k in [-8, 7] decodes back to them
    rng = np.random.default_rng(1)
    d = 96
    codes = rng.integers(-8, 8, size=d)
    scales = np.array([0.25, 0.0078125, 3.0], np.float16)   # one per group of 32
    packed = np.zeros(d // 2, np.uint8)
    for c in range(d):
        nib = codes[c] & 0xF
        packed[c // 2] |= np.uint8(nib << (4 * (c % 2)))
    m = oracle.Matrix(q=packed.reshape(1, -1), scales=scales.view(np.uint16).reshape(1, -1))
    got = oracle.decode_row(m, d, 0)
    want = codes * np.repeat(scales.astype(np.float64), 32)
    assert np.array_equal(got, want)


def test_fp16_row_decode_matches_numpy():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((3, 40)) * 0.02).astype(np.float16)
    m = oracle.Matrix(f16=w)
    for r in range(3):
        assert np.array_equal(oracle.decode_row(m, 40, r), w[r].astype(np.float64))
