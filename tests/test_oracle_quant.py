"""Pins of the oracle's block encoders / decoders: hand-worked fixtures, brute force,
round-trip bounds, identities and exact rational arithmetic."""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats as F
from oracle import quant as Q
from tests.helpers import golden_dict


def _rng(s):
    return np.random.default_rng(s)


# ------------------------------------------------------------------ nibble order
def test_nibble_order():
    codes = np.array([1, 2, 3, 4, 15, 0], np.uint8)
    assert list(Q.pack_nibbles(codes)) == [0x21, 0x43, 0x0F]
    assert np.array_equal(Q.unpack_nibbles(Q.pack_nibbles(codes)), codes)


# ------------------------------------------------------------------ NVFP4
def test_nvfp4_hand_worked_example():
    g = golden_dict("nvfp4_worked.txt")
    W = np.array([[float(v) for v in row] for row in g["x"]], np.float32)
    p = Q.nvfp4_pack(W)
    assert p["g"] == np.float32(float(g["g"][0][0]))
    assert [int(s, 16) for s in g["scales"][0]] == list(p["scales"].reshape(-1))
    exp_codes = np.array([[int(c) for c in row] for row in g["codes"]], np.uint8).reshape(-1)
    assert np.array_equal(p["codes"], exp_codes)
    packed, scales = Q.to_blobs(p)
    assert packed == bytes(int(b, 16) for b in g["packed"][0])
    assert scales[:2] == bytes([0x7E, 0x58]) and scales[2:16] == b"\0" * 14
    assert np.frombuffer(scales[16:20], np.float32)[0] == 1.0


def test_nvfp4_roundtrip_bound():
    W = _rng(3).standard_normal((64, 256)).astype(np.float32) * 0.02
    W[5, 17] = 0.9  # an outlier sets g
    p = Q.nvfp4_pack(W)
    Wh = Q.nvfp4_dequant(p)
    S = (F.e4m3_decode(p["scales"]) * p["g"]).astype(np.float64)  # [N, K/16]
    err = np.abs(W.astype(np.float64) - Wh).reshape(64, 16, 16)
    # half of the largest E2M1 gap (2) times the block scale, unless the scale underflowed
    assert np.all(err <= S[:, :, None] * 1.0 + 1e-12)
    # the block amax element decodes to within one E2M1 step of the (scaled) largest code
    blocks = W.reshape(64, 16, 16)
    i = np.argmax(np.abs(blocks), axis=2)
    ci = np.take_along_axis(p["codes"].reshape(64, 16, 16), i[:, :, None], 2)[..., 0]
    assert np.all((ci & 7) >= 6)


def test_nvfp4_zero_blocks_and_zero_tensor():
    W = np.zeros((2, 32), np.float32)
    W[1, 16:] = _rng(4).standard_normal(16).astype(np.float32)
    p = Q.nvfp4_pack(W)
    assert np.all(p["codes"].reshape(2, 32)[0] == 0) and np.all(p["codes"].reshape(2, 32)[1, :16] == 0)
    assert list(p["scales"].reshape(-1)[:3]) == [0, 0, 0]
    z = Q.nvfp4_pack(np.zeros((1, 16), np.float32))
    assert z["g"] == 1 and np.all(z["codes"] == 0) and np.all(z["scales"] == 0)
    assert np.all(Q.nvfp4_dequant(z) == 0)


def test_nvfp4_static_global_scale_saturates():
    x = np.array([[1000.0] + [0.0] * 15], np.float32)
    codes, s, g = Q.nvfp4_quantize(x, g=np.float32(0.01))
    assert g == np.float32(0.01) and s[0, 0] == 0x7E and codes[0, 0] == 7


def test_nvfp4_dequant_is_product_of_parts():
    W = _rng(5).standard_normal((8, 64)).astype(np.float32)
    p = Q.nvfp4_pack(W)
    vals = F.e2m1_decode(p["codes"]).reshape(8, 4, 16).astype(np.float64)
    sc = F.e4m3_decode(p["scales"]).astype(np.float64)[:, :, None]
    exact = vals * sc * float(p["g"])
    # the inner product e2m1 * e4m3 is exact, the outer multiply rounds once
    assert np.max(np.abs(Q.nvfp4_dequant(p).reshape(8, 4, 16) - exact) / np.maximum(np.abs(exact), 1e-30)) <= 2.0 ** -24


# ------------------------------------------------------------------ q4_0
def test_q4_0_hand_worked_example():
    g = golden_dict("q4_0_worked.txt")
    W = np.zeros((1, 64), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    p = Q.q4_0_pack(W)
    assert [int(h, 16) for h in g["d"][0]] == list(p["d"].view(np.uint16))
    c0 = [int(c) for c in g["codes0"][0]]
    c1 = [int(c) for c in g["codes1"][0]]
    exp = np.full(64, 8, np.uint8)
    exp[:len(c0)] = c0
    exp[32:32 + len(c1)] = c1
    assert np.array_equal(p["codes"], exp)
    packed, scales = Q.to_blobs(p)
    assert packed[:5] == bytes(int(b, 16) for b in g["packed0"][0])
    assert packed[16:19] == bytes(int(b, 16) for b in g["packed1"][0])
    assert scales == bytes([0x00, 0x38, 0x00, 0xB4]) + b"\0" * 12


def test_q4_0_decode_identity_all_codes():
    ds = F.fp16_round(_rng(6).standard_normal(500).astype(np.float32))
    for d in ds:
        p = dict(fmt="q4_0", N=1, K=32, codes=np.arange(32, dtype=np.uint8) % 16, d=np.array([d]))
        got = Q.q4_0_dequant(p).reshape(-1)
        exp = np.array([(q % 16 - 8) * float(d) for q in range(32)], np.float64)
        assert np.array_equal(got.astype(np.float64), exp)


def test_q4_0_roundtrip_and_idempotence():
    W = _rng(7).standard_normal((32, 128)).astype(np.float32) * 0.02
    p = Q.q4_0_pack(W)
    Wh = Q.q4_0_dequant(p)
    d = np.abs(p["d"].astype(np.float64))[:, None]
    err = np.abs(W.astype(np.float64).reshape(-1, 32) - Wh.reshape(-1, 32))
    # |err| <= |d|/2 (plus the fp16 rounding of d acting on up to 8 steps), or one step on the clamped side
    assert np.all(err <= d * 1.0 + 1e-9)
    assert np.mean(err <= d * 0.5 * (1 + 2 ** -9) * 1.02) > 0.9
    p2 = Q.q4_0_pack(Wh)
    assert np.array_equal(p2["codes"], p["codes"]) and np.array_equal(p2["d"], p["d"])


# ------------------------------------------------------------------ q8_0
def test_q8_0_hand_worked_example():
    g = golden_dict("q8_0_worked.txt")
    W = np.zeros((1, 64), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    p = Q.q8_0_pack(W)
    assert [int(h, 16) for h in g["d"][0]] == list(p["d"].view(np.uint16))
    exp = np.zeros(64, np.int8)
    exp[:len(g["codes0"][0])] = [int(c) for c in g["codes0"][0]]
    exp[32:32 + len(g["codes1"][0])] = [int(c) for c in g["codes1"][0]]
    assert np.array_equal(p["codes"], exp)


def test_q8_0_roundtrip_and_idempotence():
    W = _rng(8).standard_normal((16, 256)).astype(np.float32) * 0.02
    p = Q.q8_0_pack(W)
    Wh = Q.q8_0_dequant(p)
    d = p["d"].astype(np.float64)[:, None]
    err = np.abs(W.astype(np.float64).reshape(-1, 32) - Wh.reshape(-1, 32))
    assert np.all(err <= d * 0.5 * (1 + 2 ** -8) + 1e-12)
    assert np.array_equal(Q.q8_0_pack(Wh)["codes"], p["codes"])


def test_gguf_zero_block():
    W = np.zeros((1, 32), np.float32)
    assert np.all(Q.q4_0_pack(W)["codes"] == 8) and np.all(Q.q4_0_dequant(Q.q4_0_pack(W)) == 0)
    assert np.all(Q.q8_0_pack(W)["codes"] == 0) and np.all(Q.q8_0_dequant(Q.q8_0_pack(W)) == 0)


# ------------------------------------------------------------------ NF4
def test_nf4_codes_of_exact_codebook_values():
    cb = F.NF4_CODEBOOK
    i = np.arange(64)
    W = np.stack([cb[i % 16] * np.float32(0.5), cb[15 - i % 16] * np.float32(0.25)]).astype(np.float32)
    p = Q.nf4_pack(W)
    assert np.array_equal(p["codes"][:64], (i % 16).astype(np.uint8))
    assert np.array_equal(p["codes"][64:], (15 - i % 16).astype(np.uint8))
    assert list(p["absmax"]) == [0.5, 0.25]
    assert p["offset"] == np.float32(0.375)
    assert list(p["absmax_q"]) == [127, -127]
    assert p["s2"][0] == np.float32(0.125) / np.float32(127)
    packed, scales = Q.to_blobs(p)
    assert packed[0] == 0x10 and packed[1] == 0x32 and packed[32] == 0xEF


def test_nf4_code_is_nearest_brute_force():
    W = _rng(9).standard_normal((16, 256)).astype(np.float32) * 0.02
    W[3, :64] = 0  # an all-zero block
    p = Q.nf4_pack(W)
    cb = F.NF4_CODEBOOK.astype(np.float64)
    blocks = W.reshape(-1, 64).astype(np.float64)
    a = np.abs(blocks).max(1, keepdims=True)
    v = np.where(a == 0, 0, blocks / np.where(a == 0, 1, a))
    dist = np.abs(v[..., None] - cb)
    best = np.argmin(dist, axis=-1)
    codes = p["codes"].reshape(-1, 64)
    exact_mid = (cb[:-1] + cb[1:]) / 2
    near_mid = np.min(np.abs(v[..., None] - exact_mid), axis=-1) < 1e-6
    assert np.all((codes == best) | near_mid)
    assert np.all(codes[12] == 7)   # the zero block decodes to code 7 (value 0)


def test_nf4_midpoint_ties_go_low():
    cb = F.NF4_CODEBOOK
    mids = ((cb[:-1] + cb[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)
    W = np.zeros((1, 64), np.float32)
    W[0, 0] = 1.0
    W[0, 1:16] = mids
    W[0, 16:31] = np.nextafter(mids, np.float32(2))
    p = Q.nf4_pack(W)
    assert list(p["codes"][1:16]) == list(range(15))
    assert list(p["codes"][16:31]) == list(range(1, 16))


def test_nf4_offset_is_the_exact_mean():
    rng = _rng(10)
    # absmax values spanning a wide exponent range, where naive fp32 or fp64 summation differs
    a = np.exp2(rng.uniform(-60, 40, 5000)).astype(np.float32)
    exact = sum((Fraction(float(v)) for v in a), Fraction(0))
    total = float(exact)                      # Fraction -> float is correctly rounded
    assert np.float32(total / a.size) == Q.nf4_absmax_mean(a)
    assert math.fsum(a.astype(np.float64)) == total


def test_nf4_double_quant_bounds_and_roundtrip():
    W = _rng(11).standard_normal((64, 1280)).astype(np.float32) * 0.02
    p = Q.nf4_pack(W)
    assert p["absmax_q"].size == 64 * 20 and p["s2"].size == 5
    a_hat = Q.nf4_absmax_dequant(p)
    grp = np.arange(a_hat.size) // 256
    s2 = p["s2"][grp].astype(np.float64)
    assert np.all(np.abs(a_hat.astype(np.float64) - p["absmax"]) <= s2 * 0.5 * (1 + 1e-5) + 4e-9)
    # every group uses its full int8 range on its extreme
    for g in range(5):
        assert np.max(np.abs(p["absmax_q"][g * 256:(g + 1) * 256])) == 127
    Wh = Q.nf4_dequant(p).reshape(-1, 64).astype(np.float64)
    gap = np.max(np.diff(F.NF4_CODEBOOK.astype(np.float64))) / 2
    bound = np.abs(a_hat)[:, None] * gap + np.abs(a_hat - p["absmax"])[:, None] + 1e-9
    assert np.all(np.abs(W.reshape(-1, 64) - Wh) <= bound)


def test_nf4_ragged_dq_group():
    W = _rng(12).standard_normal((3, 64 * 100)).astype(np.float32)  # 300 blocks: groups 256 + 44
    p = Q.nf4_pack(W)
    assert p["s2"].size == 2
    packed, scales = Q.to_blobs(p)
    assert len(packed) == 3 * 6400 // 2
    assert len(scales) == 304 + 2 * 4 + 4
    assert np.frombuffer(scales[304:312], np.float32).tolist() == p["s2"].tolist()


# ------------------------------------------------------------------ activation quantiser
def test_act_quant_uses_dynamic_global_and_static_override():
    x = _rng(13).standard_normal((4, 64)).astype(np.float32)
    a = Q.quant_act_nvfp4(x)
    assert a["g"] == np.float32(np.max(np.abs(x)) / np.float32(2688))
    b = Q.quant_act_nvfp4(x, g_in=np.float32(0.5))
    assert b["g"] == np.float32(0.5)
    assert a["codes"].shape == (4, 64) and a["scales"].shape == (4, 4)
