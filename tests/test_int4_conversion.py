"""The INT4-to-fp16 code conversion used by the tensor-core FC1 loaders,
restated on the host and checked against the plain two's-complement decode
for every byte value (each fp16 pair depends on one byte of the code word).

Per pair: byte b of the sign-flipped word (n = q + 8 per nibble) is spread to
both 16-bit halves, masked to bits 0-3 (low half) and 4-7 (high half) under
the fp16 pattern of 1024, then one fp16 fma with (1, 1/16) and (-1032, -72)
gives q for both halves.  Storage follows the weight format: two codes per
byte, the low nibble is the even element.
"""
import numpy as np


def _h(bits):
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


def _fma16(a, b, c):
    # a*b + c rounded once to fp16 (the products here are exact in float64)
    return np.float16(float(a) * float(b) + float(c))


def _spread(u, b):
    byte = (u >> (8 * b)) & 0xFF
    return byte | (byte << 8) | (byte << 16) | (byte << 24)


def test_constants_are_the_intended_halves():
    assert float(_h(0x3C00)) == 1.0 and float(_h(0x2C00)) == 0.0625
    assert float(_h(0xE408)) == -1032.0 and float(_h(0xD480)) == -72.0


def test_every_byte_decodes_to_its_two_codes():
    scale = (_h(0x3C00), _h(0x2C00))
    offset = (_h(0xE408), _h(0xD480))
    for byte in range(256):
        for b in range(4):
            w = byte << (8 * b)
            u = w ^ 0x88888888
            t = (_spread(u, b) & 0x00F0000F) | 0x64006400
            lo = _fma16(_h(t & 0xFFFF), scale[0], offset[0])
            hi = _fma16(_h(t >> 16), scale[1], offset[1])
            n_even, n_odd = byte & 0xF, byte >> 4
            q_even = n_even - 16 if n_even >= 8 else n_even
            q_odd = n_odd - 16 if n_odd >= 8 else n_odd
            assert (float(lo), float(hi)) == (q_even, q_odd), (byte, b)


def test_intermediates_are_exact_fp16_values():
    # 1024 + n and 1024 + 16 n (n <= 15) and 64 + n are representable, so the
    # masked pattern and the fma introduce no rounding
    for n in range(16):
        assert float(np.float16(1024 + n)) == 1024 + n
        assert float(np.float16(1024 + 16 * n)) == 1024 + 16 * n
        assert float(np.float16((1024 + 16 * n) / 16)) == 64 + n
