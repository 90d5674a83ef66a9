"""The NVFP4 register decode's constants, checked on the host (no GPU).

The tensor-core kernels decode E2M1 codes to bf16 with byte permutes (`prmt`) from constant byte
tables, and take each E4M3 block scale as its own bit fields moved into bf16's places.  This test
reads those constants from the kernel source, emulates the byte permute by its PTX definition, and
checks against the oracle's E2M1 / E4M3 decoders, for every code:
  * eight codes -> four bf16 pairs gives each code's value (times 2^120 for the scaled table), signs
    and -0 included;
  * the scale's bit fields give its value times 2^-120 (subnormal codes onto bf16 subnormals);
  * their bf16 product, rounded to nearest even, is exactly e2m1 * e4m3 for every pair of codes.
"""
import os
import re
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "bit_weight_quantized_matmul_gb300", "csrc", "wq_tc_common.cuh")
M32 = 0xFFFFFFFF


def prmt(a, b, sel):
    """PTX prmt.b32 (default mode): byte k of the result is byte sel[4k+2:4k] of {b, a}, or that
    byte's sign replicated when sel bit 4k+3 is set; only sel[15:0] is read."""
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    out = 0
    for k in range(4):
        s = (sel >> (4 * k)) & 0xF
        byte = src[s & 7]
        if s & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        out |= byte << (8 * k)
    return out


def _body(name):
    text = open(SRC).read()
    i = text.index(name)
    return text[i:text.index("\n}\n", i)]


def _consts():
    body = _body("void e2m1x8_to_bf16(")
    h = re.search(r"H0 = X2P120 \? (0x[0-9A-Fa-f]+)u : (0x[0-9A-Fa-f]+)u, H1 = X2P120 \? (0x[0-9A-Fa-f]+)u : "
                  r"(0x[0-9A-Fa-f]+)u", body)
    lo = re.search(r"L0 = (0x[0-9A-Fa-f]+)u, L1 = (0x[0-9A-Fa-f]+)u", body)
    sign = re.findall(r"prmt\(u, u4, (0x[0-9A-Fa-f]+)u\) & (0x[0-9A-Fa-f]+)u", body)
    pair = re.findall(r"w\[(\d)\] = prmt\((lo[AB]), (hi[AB]), (0x[0-9A-Fa-f]+)u\)", body)
    mask = re.findall(r"u & (0x[0-9A-Fa-f]+)u", body)
    assert h and lo and len(sign) == 2 and len(pair) == 4 and mask, "decode constants not found"
    ints = lambda xs: [int(x, 16) for x in xs]
    H = {True: ints(h.group(1, 3)), False: ints(h.group(2, 4))}
    return H, ints(lo.groups()), [ints(s) for s in sign], [(int(w), a, b_, int(s, 16)) for w, a, b_, s in pair], \
        int(mask[0], 16)


def decode8(u, x2p120):
    """The kernel's eight-code decode, step by step with the constants from its source."""
    H, (L0, L1), signs, pairs, mask = _consts()
    H0, H1 = H[x2p120]
    sa, sb = u & mask, (u >> 16) & mask
    u4 = (u << 4) & M32
    reg = {"hiA": prmt(H0, H1, sa) | (prmt(u, u4, signs[0][0]) & signs[0][1]),
           "hiB": prmt(H0, H1, sb) | (prmt(u, u4, signs[1][0]) & signs[1][1]),
           "loA": prmt(L0, L1, sa), "loB": prmt(L0, L1, sb)}
    w = [0] * 4
    for k, a, b_, sel in pairs:
        w[k] = prmt(reg[a], reg[b_], sel)
    return w


def scale_pair(code):
    """e4m3_bf16pair_m120 on a code placed in bits 0..7 and 16..23, as the kernels place it."""
    body = _body("uint32_t e4m3_bf16pair_m120(")
    m = re.search(r"\(\(x << (\d+)\) & (0x[0-9A-Fa-f]+)u\) \| \(\(x << (\d+)\) & (0x[0-9A-Fa-f]+)u\)", body)
    assert m, "scale formula not found"
    s1, m1, s2, m2 = int(m.group(1)), int(m.group(2), 16), int(m.group(3)), int(m.group(4), 16)
    x = code | (code << 16)
    return (((x << s1) & m1) | ((x << s2) & m2)) & M32


def bf16_value(bits):
    s = -1 if bits & 0x8000 else 1
    e, m = (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return s * Fraction(m, 128) * Fraction(2) ** -126
    return s * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def round_bf16(x):
    """Round a rational to the nearest bf16 value (ties to even), subnormals included."""
    if x == 0:
        return Fraction(0)
    s, a = (-1 if x < 0 else 1), abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = a / Fraction(2) ** (max(e, -126) - 7)
    n, r = int(q), q - int(q)
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * n * Fraction(2) ** (max(e, -126) - 7)


def e2m1_exact(code):
    v = Fraction(F.E2M1_MAGNITUDES[code & 7]).limit_denominator(4)
    return -v if code & 8 else v


def decoded_codes(u, x2p120):
    w = decode8(u, x2p120)
    return [(w[k // 2] >> (16 * (k % 2))) & 0xFFFF for k in range(8)]


@pytest.mark.parametrize("x2p120", [False, True])
def test_e2m1_decode_every_code_in_every_position(x2p120):
    scale = Fraction(2) ** (120 if x2p120 else 0)
    for pos in range(8):
        for code in range(16):
            for fill in (0x00000000, 0x88888888, 0x7F7F7F7F, 0xFFFFFFFF):
                u = (fill & ~(0xF << (4 * pos)) & M32) | (code << (4 * pos))
                got = decoded_codes(u, x2p120)[pos]
                assert bf16_value(got) == e2m1_exact(code) * scale, (x2p120, pos, code, hex(fill))
                assert (got >> 15) == (code >> 3), "sign bit (-0 included)"


def test_e2m1_decode_random_words():
    rng = np.random.default_rng(7)
    for u in rng.integers(0, 1 << 32, size=3000, dtype=np.uint64):
        u = int(u)
        for x2p120 in (False, True):
            got = decoded_codes(u, x2p120)
            for k in range(8):
                code = (u >> (4 * k)) & 0xF
                assert bf16_value(got[k]) == e2m1_exact(code) * Fraction(2) ** (120 if x2p120 else 0)


def test_e4m3_scale_fields_and_products_exact():
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue  # NaN codes
        s = Fraction(float(F.e4m3_decode(np.uint8(code)))).limit_denominator(1 << 12)
        pair = scale_pair(code)
        assert pair >> 16 == pair & 0xFFFF
        assert bf16_value(pair & 0xFFFF) == s * Fraction(2) ** -120, hex(code)
        for c in range(16):
            w = decoded_codes(c, True)[0]
            assert round_bf16(bf16_value(w) * bf16_value(pair & 0xFFFF)) == e2m1_exact(c) * s, (hex(code), c)
