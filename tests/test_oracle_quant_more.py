"""Pins of the oracle's q4_1, q5_0 and FP8 E4M3 weight encoders: hand-worked fixtures, brute-force
nearest-code searches in fp64 (written independently of the encoders' rint / table search),
round-trip bounds, idempotence and torch's float8 cast."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import quant as Q
from tests.helpers import golden_dict


def _rng(s):
    return np.random.default_rng(s)


def _hex_bytes(tokens):
    return bytes(int(t, 16) for t in tokens)


# ------------------------------------------------------------------ q4_1
def _q4_1_worked():
    g = golden_dict("q4_1_worked.txt")
    W = np.zeros((1, 128), np.float32)
    W[0, :32] = float(g["rest0"][0][0])
    W[0, 32:] = float(g["rest1"][0][0])
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    return g, W


def test_q4_1_hand_worked_example():
    g, W = _q4_1_worked()
    p = Q.q4_1_pack(W)
    dm = [int(h, 16) for h in g["dm"][0]]
    assert list(p["d"].view(np.uint16)) == [dm[0], dm[2], 0, 0]
    assert list(p["m"].view(np.uint16)) == [dm[1], dm[3], 0, 0]
    c0 = [int(c) for c in g["codes0"][0]]
    c1 = [int(c) for c in g["codes1"][0]]
    assert list(p["codes"][:len(c0)]) == c0 and np.all(p["codes"][len(c0):32] == 3)
    assert list(p["codes"][32:32 + len(c1)]) == c1 and np.all(p["codes"][32 + len(c1):64] == 8)
    assert np.all(p["codes"][64:] == 0)
    packed, scales = Q.to_blobs(p)
    assert len(packed) == 80 and scales == b"\0" * 16
    assert packed[:5] == _hex_bytes(g["packed0"][0]) and packed[16:21] == _hex_bytes(g["packed1"][0])
    # the unit's side data: (d, m) of blocks 0..3 (blocks 2 and 3 of this 128-element row are zero:
    # d = m = 0)
    assert packed[64:80] == bytes([0x00, 0x3C, 0x00, 0x00, 0x00, 0x38, 0x00, 0xC4]) + b"\0" * 8


def test_q4_1_code_is_the_nearest_level_brute_force():
    """Every code minimises |(x - m) / d - q| over q = 0..15 (computed exactly with fractions on
    the fp32 quotient the reading divides); ties go to the even q."""
    W = _rng(11).standard_normal((8, 64)).astype(np.float32) * 0.02
    p = Q.q4_1_pack(W)
    b = W.reshape(-1, 32)
    for blk in range(b.shape[0]):
        d, m = np.float32(p["d"][blk]), np.float32(p["m"][blk])
        for j in range(32):
            t = np.float32(np.float32(b[blk, j] - m) / d)
            cand = sorted(range(16), key=lambda q: (abs(Fraction(float(t)) - q), q % 2))
            assert p["codes"][blk * 32 + j] == cand[0]


def test_q4_1_storage_unit_roundtrips():
    """Unpacking the 80-byte units gives back every code and every block's (d, m)."""
    p = Q.q4_1_pack(_rng(20).standard_normal((3, 256)).astype(np.float32))
    packed, _ = Q.to_blobs(p)
    u = np.frombuffer(packed, np.uint8).reshape(-1, 80)
    assert np.array_equal(Q.unpack_nibbles(u[:, :64].reshape(-1)).reshape(-1, 128), p["codes"].reshape(-1, 128))
    dm = u[:, 64:].copy().view(np.float16).reshape(-1, 2)
    assert np.array_equal(dm[:, 0].view(np.uint16), p["d"].view(np.uint16))
    assert np.array_equal(dm[:, 1].view(np.uint16), p["m"].view(np.uint16))


def test_q4_1_roundtrip_and_extremes():
    W = _rng(12).standard_normal((32, 128)).astype(np.float32) * 0.02
    p = Q.q4_1_pack(W)
    Wh = Q.q4_1_dequant(p).reshape(-1, 32).astype(np.float64)
    b = W.reshape(-1, 32).astype(np.float64)
    d = p["d"].astype(np.float64)[:, None]
    m = p["m"].astype(np.float64)[:, None]
    # half a step plus the rounding of m and d to fp16 carried over at most 15 steps
    slack = np.abs(m) * 2.0 ** -11 + 15 * d * 2.0 ** -11 + 1e-12
    assert np.all(np.abs(b - Wh) <= d / 2 + slack)
    # the block minimum maps to code 0 and decodes to m
    i = np.argmin(b, axis=1)
    assert np.all(p["codes"].reshape(-1, 32)[np.arange(b.shape[0]), i] == 0)


def test_q4_1_decode_identity_all_codes():
    for d, m in zip(F.fp16_round(_rng(13).uniform(0, 0.01, 200).astype(np.float32)),
                    F.fp16_round(_rng(14).uniform(-0.05, 0.0, 200).astype(np.float32))):
        p = dict(fmt="q4_1", N=1, K=32, codes=np.arange(32, dtype=np.uint8) % 16, d=np.array([d]), m=np.array([m]))
        got = Q.q4_1_dequant(p).reshape(-1)
        # q * d is exact in fp32; the sum with m is the exact rational sum rounded once
        exp = np.array([np.float32(float(Fraction(float(q % 16)) * Fraction(float(d)) + Fraction(float(m))))
                        for q in range(32)], np.float32)
        assert np.array_equal(got.view(np.uint32), exp.view(np.uint32))


def test_q4_1_constant_block():
    W = np.full((1, 32), 0.125, np.float32)
    p = Q.q4_1_pack(W)
    assert p["d"][0] == 0 and np.all(p["codes"] == 0) and np.all(Q.q4_1_dequant(p) == np.float32(0.125))


# ------------------------------------------------------------------ q5_0
def _q5_0_worked():
    g = golden_dict("q5_0_worked.txt")
    W = np.zeros((1, 128), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    return g, W


def test_q5_0_hand_worked_example():
    g, W = _q5_0_worked()
    p = Q.q5_0_pack(W)
    assert list(p["d"].view(np.uint16)) == [int(h, 16) for h in g["d"][0]]
    c = p["codes"]
    c0 = [int(v) for v in g["codes0"][0]]
    c1 = [int(v) for v in g["codes1"][0]]
    assert list(c[:len(c0)]) == c0 and np.all(c[len(c0):32] == 16)
    assert list(c[32:32 + len(c1)]) == c1 and np.all(c[32 + len(c1):] == 16)
    packed, scales = Q.to_blobs(p)
    assert len(packed) == 80
    n0 = _hex_bytes(g["nibbles0"][0])
    n1 = _hex_bytes(g["nibbles1"][0])
    assert packed[:len(n0)] == n0 and packed[len(n0):16] == b"\0" * (16 - len(n0))
    assert packed[16:16 + len(n1)] == n1 and packed[16 + len(n1):64] == b"\0" * (48 - len(n1))
    assert packed[64:80] == _hex_bytes(g["highbits"][0])
    assert scales == bytes([0x00, 0x3C, 0x00, 0xB8, 0x00, 0x80, 0x00, 0x80]) + b"\0" * 8


def test_q5_0_code_is_the_nearest_level_brute_force():
    W = _rng(15).standard_normal((4, 128)).astype(np.float32) * 0.02
    p = Q.q5_0_pack(W)
    b = W.reshape(-1, 32)
    for blk in range(b.shape[0]):
        d = np.float32(p["d"][blk])
        for j in range(32):
            t = Fraction(float(np.float32(b[blk, j] / d)))
            cand = sorted(range(32), key=lambda q: (abs(t - (q - 16)), q % 2))
            assert p["codes"][blk * 32 + j] == cand[0]


def test_q5_0_roundtrip_and_idempotence():
    W = _rng(16).standard_normal((16, 256)).astype(np.float32) * 0.02
    p = Q.q5_0_pack(W)
    Wh = Q.q5_0_dequant(p)
    d = np.abs(p["d"].astype(np.float64))[:, None]
    err = np.abs(W.astype(np.float64).reshape(-1, 32) - Wh.reshape(-1, 32).astype(np.float64))
    assert np.all(err <= d * 1.0 + 1e-12)
    p2 = Q.q5_0_pack(Wh)
    assert np.array_equal(p2["codes"], p["codes"]) and np.array_equal(p2["d"], p["d"])


def test_q5_0_storage_unit_roundtrips():
    """Unpacking the storage unit (nibbles + fifth-bit plane) gives back every code."""
    p = Q.q5_0_pack(_rng(17).standard_normal((3, 256)).astype(np.float32))
    packed, _ = Q.to_blobs(p)
    u = np.frombuffer(packed, np.uint8).reshape(-1, 80)
    lo = Q.unpack_nibbles(u[:, :64].reshape(-1)).reshape(-1, 128)
    hi = np.unpackbits(u[:, 64:], axis=1, bitorder="little")
    assert np.array_equal(lo | (hi << 4), p["codes"].reshape(-1, 128))


# ------------------------------------------------------------------ FP8 E4M3
def test_fp8_hand_worked_example():
    g = golden_dict("fp8_worked.txt")
    W = np.zeros((4, 32), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    W[0, :len(x0)] = x0
    W[1] = W[0] * 2
    x3 = [float(v) for v in g["x3"][0]]
    W[3, :len(x3)] = x3
    W[0, 10] = -0.0
    p = Q.fp8_pack(W)
    assert list(p["s"][:3]) == [float(v) for v in g["s"][0]]
    c = p["codes"].reshape(4, 32)
    c0 = [int(v, 16) for v in g["codes0"][0]]
    c3 = [int(v, 16) for v in g["codes3"][0]]
    assert list(c[0, :len(c0)]) == c0 and np.all(c[0, len(c0):] == 0)
    assert np.array_equal(c[1], c[0]) and np.all(c[2] == 0)
    assert list(c[3, :len(c3)]) == c3
    packed, scales = Q.to_blobs(p)
    assert len(packed) == 128 and len(scales) == 16


def test_fp8_codes_match_torch_cast_of_the_scaled_values():
    W = _rng(18).standard_normal((64, 256)).astype(np.float32) * 0.02
    W[3, 7] = 0.4
    p = Q.fp8_pack(W)
    ratio = (W / p["s"][:, None]).astype(np.float32)
    assert np.max(np.abs(ratio)) < 464
    ref = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(-1)
    assert np.array_equal(ref, p["codes"])
    # each row's amax element is the top code (+-448)
    i = np.argmax(np.abs(W), axis=1)
    assert np.all((p["codes"].reshape(64, 256)[np.arange(64), i] & 0x7F) == 0x7E)


def test_fp8_roundtrip_bound_and_decode():
    W = _rng(19).standard_normal((16, 128)).astype(np.float32) * 0.02
    p = Q.fp8_pack(W)
    Wh = Q.fp8_dequant(p).astype(np.float64)
    s = p["s"].astype(np.float64)[:, None]
    # E4M3 keeps 4 significant bits: |w/s - e4m3| <= 2^-4 |w/s| for normals, <= 2^-10 below 2^-6
    r = np.abs(W.astype(np.float64) / s)
    bound = s * np.maximum(r * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20) + np.abs(Wh) * 2.0 ** -24
    assert np.all(np.abs(W - Wh) <= bound)
    v = F.e4m3_decode(p["codes"]).reshape(16, 128).astype(np.float64)
    assert np.array_equal(Wh, (v * s).astype(np.float32).astype(np.float64))
