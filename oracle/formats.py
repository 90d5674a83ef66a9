"""Scalar number formats of the quantised weights and activations (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources
-------
* NVFP4 element and scale types: model card "whisper-large-v3-turbo -- NVFP4",
  section "What is quantized" (FP4 E2M1 values, an FP8 E4M3 scale per 16
  values, one FP32 global scale per module); PR "asr: add a 4-bit nvfp4 option
  for cards short of VRAM", summary (E2M1 in blocks of 16, fp8 scale per
  block).  The pages name the types but print no tables; the value sets are
  those of the OCP Microscaling Formats spec v1.0 (E2M1) and the OCP 8-bit
  floating point spec (E4M3, the "fn" variant: no infinities, one NaN
  mantissa pattern, max 448).
* fp16 block scale of q4_0 / q8_0: PR "Run quantized Whisper on the fused
  Metal decode path", section "Summary" (GGUF q8_0 / q4_0); binary16 is IEEE.
* NF4 codebook: PR "asr: add a 4-bit nf4 option for the Whisper engine",
  sections "summary" and "What's here" (bitsandbytes NF4).  The values are the
  4-bit NormalFloat data type of Dettmers et al. 2023 (QLoRA), section 3, whose
  appendix prints the 16 values used below.

Rounding rules (readings where the pages are silent)
----------------------------------------------------
* Every encoder rounds to nearest, ties to the even code, and saturates to the
  largest finite magnitude ("satfinite").
* E2M1 takes its sign from the sign bit of the input, so a small negative
  value that rounds to zero is stored as code 8 (-0).
"""

import numpy as np

# --------------------------------------------------------------------------
# E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf / NaN.
# Codes 0..7 hold the magnitudes below; bit 3 is the sign.
# --------------------------------------------------------------------------
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)


def e2m1_decode(code):
    """uint8 code (0..15) -> float32 value, by the E2M1 definition."""
    c = np.asarray(code).astype(np.int64) & 0xF
    e = (c >> 1) & 3
    m = c & 1
    # e == 0: subnormal m * 2^-1 ; otherwise (1 + m/2) * 2^(e-1)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(c >> 3 == 1, -mag, mag).astype(np.float32)


def _nearest_code_ties_even(a, table):
    """Index of the entry of the increasing ``table`` nearest to ``a`` >= 0.

    Distances are compared exactly (fp64 holds every difference of an fp32
    input and a table value).  Ties go to the even index.  Inputs above the
    last entry saturate to it.
    """
    a = np.asarray(a, np.float64)
    hi = np.searchsorted(table, a, side="left")  # first entry >= a
    hi = np.minimum(hi, len(table) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    pick_hi = np.where(d_hi < d_lo, True, np.where(d_hi > d_lo, False, hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    idx = np.where(a >= table[-1], len(table) - 1, idx)
    return idx.astype(np.int64)


def e2m1_encode(x):
    """float32 -> uint8 E2M1 code, round to nearest even, saturate at 6."""
    x = np.asarray(x, np.float32)
    mag = _nearest_code_ties_even(np.abs(x).astype(np.float64), E2M1_MAGNITUDES)
    sign = np.signbit(x).astype(np.int64)
    return (mag | (sign << 3)).astype(np.uint8)


# --------------------------------------------------------------------------
# E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits.  exp=0 is
# subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinities; max 448.
# --------------------------------------------------------------------------
def e4m3_decode(byte):
    """uint8 -> float32 value by the E4M3 definition (NaN for 0x7F / 0xFF)."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    s = b >> 7
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float32)


# every finite non-negative E4M3 value, in code order 0x00..0x7E (increasing)
E4M3_FINITE_POS = e4m3_decode(np.arange(0x7F)).astype(np.float64)
E4M3_MAX = 448.0


def e4m3_encode_satfinite(x):
    """float32 -> uint8 E4M3 code: nearest value, ties to even code, |x| >= 448 -> 448.

    The sign bit is copied from the input (the block scales it encodes are
    never negative).
    """
    x = np.asarray(x, np.float32)
    mag = _nearest_code_ties_even(np.abs(x).astype(np.float64), E4M3_FINITE_POS)
    sign = np.signbit(x).astype(np.int64)
    return (mag | (sign << 7)).astype(np.uint8)


# --------------------------------------------------------------------------
# IEEE binary16 (block scale d of q4_0 / q8_0).  numpy's float32 -> float16
# conversion rounds to nearest even (pinned against torch in the tests).
# --------------------------------------------------------------------------
def fp16_round(x):
    """float32 -> float16 (round to nearest even)."""
    return np.asarray(x, np.float32).astype(np.float16)


def bf16_bits_to_f32(bits):
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


# --------------------------------------------------------------------------
# NF4 codebook (QLoRA, appendix table).  Index 0 = -1, index 7 = 0,
# index 15 = +1; 7 negative and 8 positive normal quantiles scaled to [-1, 1].
# --------------------------------------------------------------------------
NF4_CODEBOOK = np.array([
    -1.0,
    -0.6961928009986877,
    -0.5250730514526367,
    -0.39491748809814453,
    -0.28444138169288635,
    -0.18477343022823334,
    -0.09105003625154495,
    0.0,
    0.07958029955625534,
    0.16093020141124725,
    0.24611230194568634,
    0.33791524171829224,
    0.44070982933044434,
    0.5626170039176941,
    0.7229568362236023,
    1.0,
], dtype=np.float32)


def nf4_construction_fp64():
    """The NormalFloat construction of QLoRA section 3, evaluated in fp64.

    Quantiles of N(0, 1): the positive half uses 8 probabilities evenly spaced
    from delta down to 1/2 (1/2 itself excluded), the negative half 7, where
    delta = ((1 - 1/30) + (1 - 1/32)) / 2 is the mean of the inner quantile
    offsets for 15 and 16 bins; the shared zero is kept once and the set is
    divided by its largest value.  Used only to pin ``NF4_CODEBOOK``.
    """
    from scipy.special import ndtri

    delta = 0.5 * ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0))
    pos = ndtri(np.linspace(delta, 0.5, 9)[:-1])
    neg = -ndtri(np.linspace(delta, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([neg, [0.0], pos]))
    return v / v.max()
