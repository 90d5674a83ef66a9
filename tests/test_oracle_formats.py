"""Pins of the oracle's scalar formats against closed forms, spec tables and torch casts."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.helpers import golden_lines


# ------------------------------------------------------------------ E2M1
def test_e2m1_decode_exhaustive_vs_spec_table():
    rows = golden_lines("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = F.e2m1_decode(np.uint8(int(code)))
        assert float(got) == float(val)
        assert np.signbit(got) == val.startswith("-")


@pytest.mark.parametrize("x,code", [
    (0.0, 0), (0.24, 0), (0.25, 0), (0.26, 1), (0.5, 1), (0.74, 1), (0.75, 2), (1.0, 2),
    (1.25, 2), (1.26, 3), (1.5, 3), (1.74, 3), (1.75, 4), (2.0, 4), (2.5, 4), (2.51, 5),
    (3.0, 5), (3.49, 5), (3.5, 6), (4.0, 6), (5.0, 6), (5.01, 7), (6.0, 7), (7.0, 7),
    (1e30, 7), (float("inf"), 7), (-0.25, 8), (-0.0, 8), (-0.3, 9), (-5.0, 14), (-100.0, 15),
])
def test_e2m1_encode_ties_even_and_saturation(x, code):
    assert int(F.e2m1_encode(np.float32(x))) == code


def test_e2m1_encode_is_nearest_on_a_fine_grid():
    xs = np.linspace(-7, 7, 20001).astype(np.float32)
    codes = F.e2m1_encode(xs)
    vals = F.e2m1_decode(codes).astype(np.float64)
    allv = F.e2m1_decode(np.arange(16)).astype(np.float64)
    best = np.min(np.abs(xs[:, None].astype(np.float64).clip(-6, 6) - allv[None, :]), axis=1)
    assert np.all(np.abs(xs.astype(np.float64).clip(-6, 6) - vals) == best)


def test_e2m1_decode_matches_torch_fp4_view_when_available():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("torch has no fp4 dtype")
    packed = torch.arange(256, dtype=torch.uint8)
    try:
        pairs = packed.view(torch.float4_e2m1fn_x2)
        _ = pairs.to(torch.float32)
    except Exception:
        pytest.skip("torch cannot widen float4_e2m1fn_x2 on this build")
    lo = F.e2m1_decode(packed.numpy() & 0xF)
    hi = F.e2m1_decode(packed.numpy() >> 4)
    t = pairs.to(torch.float32).numpy().reshape(-1)
    assert np.array_equal(np.stack([lo, hi], 1).reshape(-1), t)


# ------------------------------------------------------------------ E4M3
def test_e4m3_decode_spec_table():
    for code, val in golden_lines("e4m3_values.txt"):
        got = float(F.e4m3_decode(np.uint8(int(code, 16))))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), code


def test_e4m3_decode_all_256_vs_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = F.e4m3_decode(b.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(1)
    # random magnitudes across the whole range, every code value, and every midpoint
    r = np.exp2(rng.uniform(-12, np.log2(460), 200000)).astype(np.float32)
    vals = F.E4M3_FINITE_POS
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    xs = np.concatenate([r, vals.astype(np.float32), mids,
                         np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    xs = xs[xs < 464]
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.e4m3_encode_satfinite(xs)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates():
    xs = np.array([448, 463.9, 464, 465, 480, 1e6, 3e38, np.inf], np.float32)
    assert np.all(F.e4m3_encode_satfinite(xs) == 0x7E)
    assert int(F.e4m3_encode_satfinite(np.float32(2.0 ** -10))) == 0          # tie 0 / 2^-9 -> even 0
    assert int(F.e4m3_encode_satfinite(np.float32(3 * 2.0 ** -10))) == 2     # tie 1 / 2 -> even 2
    assert int(F.e4m3_encode_satfinite(np.float32(1.0625))) == 0x38          # tie 1 / 1.125 -> 1


# ------------------------------------------------------------------ fp16
def test_fp16_round_vs_torch():
    rng = np.random.default_rng(2)
    xs = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 0.02,
        np.exp2(rng.uniform(-26, 16, 100000)).astype(np.float32),
        # exact ties between neighbouring fp16 values, including subnormals
        ((np.arange(1, 4000, dtype=np.float64) + 0.5) * 2.0 ** -24).astype(np.float32),
        ((np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -10).astype(np.float32),
    ])
    ref = torch.from_numpy(xs).to(torch.float16).numpy()
    got = F.fp16_round(xs)
    assert np.array_equal(ref.view(np.uint16), got.view(np.uint16))


def test_bf16_widening():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    got = F.bf16_bits_to_f32(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])


# ------------------------------------------------------------------ NF4 codebook
def test_nf4_codebook_matches_printed_table():
    t = np.array([float(r[0]) for r in golden_lines("nf4_codebook.txt")], np.float32)
    assert np.array_equal(t.view(np.uint32), F.NF4_CODEBOOK.view(np.uint32))


def test_nf4_codebook_invariants():
    c = F.NF4_CODEBOOK
    assert c.dtype == np.float32 and c.size == 16
    assert np.all(np.diff(c) > 0)
    assert c[0] == -1 and c[7] == 0 and c[15] == 1
    assert np.sum(c < 0) == 7 and np.sum(c > 0) == 8


def test_nf4_codebook_follows_normalfloat_construction():
    v = F.nf4_construction_fp64()
    # within a few fp32 ulps of the construction evaluated in fp64
    assert np.max(np.abs(v - F.NF4_CODEBOOK.astype(np.float64))) < 4 * 2.0 ** -24 * 2
    # and the construction really is built from normal quantiles: the positive half
    # is asymmetric to the negative half (8 values against 7)
    assert not np.allclose(-v[1:7], v[9:15])
