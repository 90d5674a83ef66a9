"""Block encoders and decoders of the quantised weight formats (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Every matrix is PyTorch-Linear shaped, W[N, K] row-major with K contiguous,
and every quantisation block runs along K.  All steps are float32 IEEE
operations in the order written here; ``np.rint`` rounds half to even.

Formats and the passages they follow
------------------------------------
* NF4 with double-quantised absmax -- PR "asr: add a 4-bit nf4 option for the
  Whisper engine", "What's here" (NF4, double-quant, bf16 compute); block 64,
  second level 8-bit over groups of 256 absmax values with an fp32 scale.
  Readings (the pages print no formula): codes use the exact fp32 absmax; the
  second level subtracts the mean of all absmax values (QLoRA section 3) and
  quantises the centred values to symmetric int8.
* NVFP4 -- model card "whisper-large-v3-turbo -- NVFP4", "What is quantized";
  PR "asr: add a 4-bit nvfp4 option", summary.  E2M1 codes in blocks of 16
  along K, one E4M3 scale per block, one fp32 global scale per tensor.
  Reading: the global value g is stored as the decode multiplier
  g = amax / (6 * 448), so that x ~ e2m1 * e4m3 * g.
* NVFP4 activations -- same model card, "What is quantized" (activations
  quantised per 16-value group at runtime) and "Honest summary" (W4A4 on
  Blackwell).  Reading: the per-tensor g comes from the dynamic amax unless a
  static one is supplied.
* q4_0 / q8_0 -- PR "Run quantized Whisper on the fused Metal decode path",
  "Summary" and "Why the policy".  Blocks of 32 with an fp16 scale d;
  q4_0 decodes as (q - 8) * d, q8_0 as q * d.  Readings: the codes are
  computed against the stored (fp16-rounded) d; q4_0's d maps the block's
  signed extreme to code 0 (d = extreme / -8).
* q4_1 / q5_0 -- the same PR, "Why the policy" (the other GGUF block types,
  slower there without fast kernels).  The pages name them only.  Readings:
  GGUF's block definitions, blocks of 32 with fp16 scales: q4_1 stores d and
  a minimum m and decodes as q * d + m (q in 0..15, d = (max - min) / 15,
  m = min); q5_0 stores d and 5-bit codes and decodes as (q - 16) * d
  (d = extreme / -16, the q4_0 rule with 16 levels a side).  Codes are
  computed against the stored fp16 values, rounding half to even.
* FP8 E4M3 weights -- model card "whisper-large-v3-turbo -- NVFP4", "Honest
  summary" and "Why the encoder/decoder split matters" (the FP8 build and the
  NVFP4-encoder / FP8-decoder build).  The card names the type only.
  Reading: E4M3 codes with one fp32 scale per output row (weight row of W),
  s = amax_row / 448, code = E4M3(w / s) round to nearest even, saturating;
  decode E4M3(code) * s.
"""

import math

import numpy as np

from . import formats as F

NF4_BLOCK = 64
NF4_DQ_GROUP = 256
NVFP4_BLOCK = 16
GGUF_BLOCK = 32
E2M1_MAX = np.float32(6.0)
NVFP4_GLOBAL_DIV = np.float32(6.0 * 448.0)  # 2688, exact


def _f32(x):
    return np.asarray(x, np.float32)


# ---------------------------------------------------------------- nibbles
def pack_nibbles(codes):
    """Element 2j goes to the low nibble of byte j, element 2j+1 to the high."""
    c = np.asarray(codes, np.uint8).reshape(-1)
    assert c.size % 2 == 0
    return (c[0::2] & 0xF) | ((c[1::2] & 0xF) << 4)


def unpack_nibbles(packed):
    p = np.asarray(packed, np.uint8).reshape(-1)
    out = np.empty(p.size * 2, np.uint8)
    out[0::2] = p & 0xF
    out[1::2] = p >> 4
    return out


# ---------------------------------------------------------------- NF4
def nf4_absmax_mean(absmax):
    """Mean of the absmax values: exact sum rounded once to fp64 (math.fsum),
    divided by the count in fp64, rounded once to fp32."""
    total = math.fsum(np.asarray(absmax, np.float64).tolist())
    return np.float32(total / absmax.size)


def nf4_pack(W):
    """W float32 [N, K] (K % 64 == 0) -> dict of NF4 codes and double-quantised absmax."""
    W = _f32(W)
    N, K = W.shape
    assert K % NF4_BLOCK == 0
    blocks = W.reshape(-1, NF4_BLOCK)
    # step 1: block absmax (exact in fp32)
    absmax = np.max(np.abs(blocks), axis=1).astype(np.float32)
    # step 2: normalise by the block absmax (one fp32 division); an all-zero block maps to 0
    safe = np.where(absmax == 0, np.float32(1), absmax)
    v = np.where(absmax[:, None] == 0, np.float32(0), blocks / safe[:, None]).astype(np.float32)
    # step 3: code = number of codebook midpoints strictly below v (ties go to the lower code)
    cb = F.NF4_CODEBOOK
    mids = ((cb[:-1] + cb[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)
    codes = np.sum(v[:, :, None] > mids[None, None, :], axis=2).astype(np.uint8)

    # double quantisation of the absmax values
    offset = nf4_absmax_mean(absmax)
    centred = (absmax - offset).astype(np.float32)
    nb = absmax.size
    ng = (nb + NF4_DQ_GROUP - 1) // NF4_DQ_GROUP
    s2 = np.zeros(ng, np.float32)
    q = np.zeros(nb, np.int8)
    for g in range(ng):
        t = centred[g * NF4_DQ_GROUP:(g + 1) * NF4_DQ_GROUP]
        s = np.float32(np.max(np.abs(t)) / np.float32(127))
        s2[g] = s
        if s != 0:
            q[g * NF4_DQ_GROUP:(g + 1) * NF4_DQ_GROUP] = np.clip(np.rint(t / s), -127, 127).astype(np.int8)
    return dict(fmt="nf4", N=N, K=K, codes=codes.reshape(-1), absmax=absmax,
                absmax_q=q, s2=s2, offset=offset)


def nf4_absmax_dequant(p):
    """Second-level decode: a_hat = q * s2 + offset, two fp32 roundings (no FMA)."""
    grp = np.arange(p["absmax_q"].size) // NF4_DQ_GROUP
    prod = (p["absmax_q"].astype(np.float32) * p["s2"][grp]).astype(np.float32)
    return (prod + p["offset"]).astype(np.float32)


def nf4_dequant(p):
    a_hat = nf4_absmax_dequant(p)
    vals = F.NF4_CODEBOOK[p["codes"]].reshape(-1, NF4_BLOCK)
    return (vals * a_hat[:, None]).astype(np.float32).reshape(p["N"], p["K"])


# ---------------------------------------------------------------- NVFP4
def nvfp4_global(amax):
    """Decode multiplier g = amax / 2688 (fp32 division); g = 1 for an all-zero tensor."""
    amax = np.float32(amax)
    return np.float32(1) if amax == 0 else np.float32(amax / NVFP4_GLOBAL_DIV)


def nvfp4_quantize(X, g=None):
    """X float32 [R, C] (C % 16 == 0) -> E2M1 codes [R, C], E4M3 scales [R, C/16], g.

    Per 16-block: s = e4m3((amax_b / 6) / g), S = dec(s) * g, code = e2m1(x / S),
    with code 0 where S == 0.  ``g`` is the per-tensor decode multiplier; when
    it is None it comes from the tensor's own amax.
    """
    X = _f32(X)
    R, C = X.shape
    assert C % NVFP4_BLOCK == 0
    if g is None:
        g = nvfp4_global(np.max(np.abs(X)) if X.size else 0)
    g = np.float32(g)
    xb = X.reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(xb), axis=2).astype(np.float32)
    ratio = ((amax_b / E2M1_MAX).astype(np.float32) / g).astype(np.float32)
    s = F.e4m3_encode_satfinite(ratio)
    S = (F.e4m3_decode(s) * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        scaled = (xb / S[:, :, None]).astype(np.float32)
    codes = np.where(S[:, :, None] == 0, np.uint8(0), F.e2m1_encode(scaled)).astype(np.uint8)
    return codes.reshape(R, C), s, g


def nvfp4_dequant_parts(codes, scales, g):
    """x_hat = (e2m1(code) * e4m3(s)) * g: the inner product is exact, the outer rounds once."""
    codes = np.asarray(codes, np.uint8)
    R, C = codes.shape
    inner = (F.e2m1_decode(codes).reshape(R, C // NVFP4_BLOCK, NVFP4_BLOCK)
             * F.e4m3_decode(scales)[:, :, None]).astype(np.float32)
    return (inner * np.float32(g)).astype(np.float32).reshape(R, C)


def nvfp4_pack(W):
    codes, s, g = nvfp4_quantize(W)
    N, K = codes.shape
    return dict(fmt="nvfp4", N=N, K=K, codes=codes.reshape(-1), scales=s, g=g)


def nvfp4_dequant(p):
    return nvfp4_dequant_parts(p["codes"].reshape(p["N"], p["K"]), p["scales"], p["g"])


def quant_act_nvfp4(x, g_in=None):
    """Runtime activation quantiser of W4A4 mode: the same block encoder applied to
    x [M, K] (bf16 values widened to fp32), per 16 along K, with a dynamic per-tensor
    g unless ``g_in`` is given."""
    codes, s, g = nvfp4_quantize(x, g_in)
    return dict(codes=codes, scales=s, g=g)


# ---------------------------------------------------------------- q4_0
def q4_0_pack(W):
    W = _f32(W)
    N, K = W.shape
    assert K % GGUF_BLOCK == 0
    b = W.reshape(-1, GGUF_BLOCK)
    idx = np.argmax(np.abs(b), axis=1)            # first index of the largest |x|
    extreme = b[np.arange(b.shape[0]), idx]
    d = F.fp16_round((extreme / np.float32(-8)).astype(np.float32))
    dq = d.astype(np.float32)
    safe = np.where(dq == 0, np.float32(1), dq)
    q = np.clip(np.rint((b / safe[:, None]).astype(np.float32)) + 8, 0, 15)
    q = np.where(dq[:, None] == 0, 8, q).astype(np.uint8)
    return dict(fmt="q4_0", N=N, K=K, codes=q.reshape(-1), d=d)


def q4_0_dequant(p):
    q = p["codes"].astype(np.float32).reshape(-1, GGUF_BLOCK)
    dq = p["d"].astype(np.float32)
    return ((q - np.float32(8)) * dq[:, None]).astype(np.float32).reshape(p["N"], p["K"])


# ---------------------------------------------------------------- q8_0
def q8_0_pack(W):
    W = _f32(W)
    N, K = W.shape
    assert K % GGUF_BLOCK == 0
    b = W.reshape(-1, GGUF_BLOCK)
    amax = np.max(np.abs(b), axis=1).astype(np.float32)
    d = F.fp16_round((amax / np.float32(127)).astype(np.float32))
    dq = d.astype(np.float32)
    safe = np.where(dq == 0, np.float32(1), dq)
    q = np.clip(np.rint((b / safe[:, None]).astype(np.float32)), -127, 127)
    q = np.where(dq[:, None] == 0, 0, q).astype(np.int8)
    return dict(fmt="q8_0", N=N, K=K, codes=q.reshape(-1), d=d)


def q8_0_dequant(p):
    q = p["codes"].astype(np.float32).reshape(-1, GGUF_BLOCK)
    return (q * p["d"].astype(np.float32)[:, None]).astype(np.float32).reshape(p["N"], p["K"])


# ---------------------------------------------------------------- q4_1
def q4_1_pack(W):
    """Blocks of 32: m = fp16(min), d = fp16((max - min) / 15), q = clamp(rint((x - m) / d), 0, 15)
    with the stored m and d (q = 0 where d == 0)."""
    W = _f32(W)
    N, K = W.shape
    assert K % GGUF_BLOCK == 0
    b = W.reshape(-1, GGUF_BLOCK)
    mn = np.min(b, axis=1).astype(np.float32)
    mx = np.max(b, axis=1).astype(np.float32)
    d = F.fp16_round(((mx - mn).astype(np.float32) / np.float32(15)).astype(np.float32))
    m = F.fp16_round(mn)
    dq, mq = d.astype(np.float32), m.astype(np.float32)
    safe = np.where(dq == 0, np.float32(1), dq)
    t = (b - mq[:, None]).astype(np.float32)
    q = np.clip(np.rint((t / safe[:, None]).astype(np.float32)), 0, 15)
    q = np.where(dq[:, None] == 0, 0, q).astype(np.uint8)
    return dict(fmt="q4_1", N=N, K=K, codes=q.reshape(-1), d=d, m=m)


def q4_1_dequant(p):
    """x_hat = q * d + m: the product is exact in fp32 (4-bit q, 11-bit d), the sum rounds once."""
    q = p["codes"].astype(np.float32).reshape(-1, GGUF_BLOCK)
    prod = (q * p["d"].astype(np.float32)[:, None]).astype(np.float32)
    return (prod + p["m"].astype(np.float32)[:, None]).astype(np.float32).reshape(p["N"], p["K"])


# ---------------------------------------------------------------- q5_0
def q5_0_pack(W):
    """Blocks of 32: d = fp16(extreme / -16) with the extreme the first element of largest |x|,
    q = clamp(rint(x / d) + 16, 0, 31) with the stored d (q = 16 where d == 0)."""
    W = _f32(W)
    N, K = W.shape
    assert K % GGUF_BLOCK == 0
    b = W.reshape(-1, GGUF_BLOCK)
    idx = np.argmax(np.abs(b), axis=1)
    extreme = b[np.arange(b.shape[0]), idx]
    d = F.fp16_round((extreme / np.float32(-16)).astype(np.float32))
    dq = d.astype(np.float32)
    safe = np.where(dq == 0, np.float32(1), dq)
    q = np.clip(np.rint((b / safe[:, None]).astype(np.float32)) + 16, 0, 31)
    q = np.where(dq[:, None] == 0, 16, q).astype(np.uint8)
    return dict(fmt="q5_0", N=N, K=K, codes=q.reshape(-1), d=d)


def q5_0_dequant(p):
    q = p["codes"].astype(np.float32).reshape(-1, GGUF_BLOCK)
    return ((q - np.float32(16)) * p["d"].astype(np.float32)[:, None]).astype(np.float32).reshape(p["N"], p["K"])


# ---------------------------------------------------------------- FP8 E4M3 weights
FP8_MAX = np.float32(448.0)


def fp8_pack(W):
    """One fp32 scale per row s = amax_row / 448 (fp32 division); code = E4M3(w / s), round to nearest
    even, saturating, sign copied; code 0 where s == 0."""
    W = _f32(W)
    N, K = W.shape
    amax = np.max(np.abs(W), axis=1).astype(np.float32) if K else np.zeros(N, np.float32)
    s = (amax / FP8_MAX).astype(np.float32)
    safe = np.where(s == 0, np.float32(1), s)
    codes = F.e4m3_encode_satfinite((W / safe[:, None]).astype(np.float32))
    codes = np.where(s[:, None] == 0, np.uint8(0), codes).astype(np.uint8)
    return dict(fmt="fp8", N=N, K=K, codes=codes.reshape(-1), s=s)


def fp8_dequant(p):
    """x_hat = E4M3(code) * s: one fp32 rounding."""
    v = F.e4m3_decode(p["codes"]).reshape(p["N"], p["K"])
    return (v * p["s"][:, None]).astype(np.float32)


# ---------------------------------------------------------------- dispatch
PACK = {"nf4": nf4_pack, "nvfp4": nvfp4_pack, "q4_0": q4_0_pack, "q8_0": q8_0_pack,
        "q4_1": q4_1_pack, "q5_0": q5_0_pack, "fp8": fp8_pack}
DEQUANT = {"nf4": nf4_dequant, "nvfp4": nvfp4_dequant, "q4_0": q4_0_dequant, "q8_0": q8_0_dequant,
           "q4_1": q4_1_dequant, "q5_0": q5_0_dequant, "fp8": fp8_dequant}


# ---------------------------------------------------------------- byte blobs
def _align16(n):
    return (n + 15) // 16 * 16


def to_blobs(p):
    """The (packed, scales) byte strings of the library's storage layout.

    packed: nf4 / nvfp4 / q4_0: two codes per byte (element 2j in the low nibble);
            q8_0: one int8 per element.
    scales: nf4:   int8 absmax codes [N*K/64] | zero pad to 16 B | fp32 s2 [groups] | fp32 offset
            nvfp4: E4M3 bytes [N, K/16] row-major | zero pad to 16 B | fp32 g
            q4_0 / q8_0 / q5_0: fp16 d [N*K/32] | zero pad to 16 B
            q4_1:  16 zero bytes (its scales are inside the packed units)
            fp8:   fp32 s [N] | zero pad to 16 B
    q5_0 / q4_1 packed: 80-byte units, one per 128 consecutive elements of a row: 64 bytes of
            (low) nibbles, element 2j in the low nibble of byte j, then 16 bytes of side data --
            q5_0: the fifth bits (bit j of byte i is the fifth bit of element 8i + j);
            q4_1: the four blocks' (fp16 d, fp16 m) pairs, GGUF keeping a block's scales
            beside its codes.
    """
    fmt = p["fmt"]
    if fmt in ("nf4", "nvfp4", "q4_0"):
        packed = pack_nibbles(p["codes"]).tobytes()
    elif fmt == "q5_0":
        assert p["K"] % 128 == 0, "q5_0 rows hold whole 128-element units"
        c = np.asarray(p["codes"], np.uint8).reshape(-1, 128)
        lo = pack_nibbles(c & 0xF).reshape(-1, 64)
        hi = np.packbits((c >> 4).astype(np.uint8).reshape(-1, 16, 8), axis=2, bitorder="little").reshape(-1, 16)
        packed = np.concatenate([lo, hi], axis=1).tobytes()
    elif fmt == "q4_1":
        assert p["K"] % 128 == 0, "q4_1 rows hold whole 128-element units"
        c = np.asarray(p["codes"], np.uint8).reshape(-1, 128)
        lo = pack_nibbles(c).reshape(-1, 64)
        dm = np.stack([np.asarray(p["d"], np.float16), np.asarray(p["m"], np.float16)], axis=1)
        packed = np.concatenate([lo, dm.reshape(-1, 8).view(np.uint8)], axis=1).tobytes()
    elif fmt == "q8_0":
        packed = np.asarray(p["codes"], np.int8).tobytes()
    else:  # fp8
        packed = np.asarray(p["codes"], np.uint8).tobytes()
    if fmt == "nf4":
        a = np.asarray(p["absmax_q"], np.int8).tobytes()
        scales = a + b"\0" * (_align16(len(a)) - len(a))
        scales += np.asarray(p["s2"], np.float32).tobytes() + np.float32(p["offset"]).tobytes()
    elif fmt == "nvfp4":
        s = np.asarray(p["scales"], np.uint8).tobytes()
        scales = s + b"\0" * (_align16(len(s)) - len(s)) + np.float32(p["g"]).tobytes()
    elif fmt == "q4_1":
        scales = b"\0" * 16  # the (d, m) pairs travel inside the packed units
    elif fmt == "fp8":
        sv = np.asarray(p["s"], np.float32).tobytes()
        scales = sv + b"\0" * (_align16(len(sv)) - len(sv))
    else:
        d = np.asarray(p["d"], np.float16).tobytes()
        scales = d + b"\0" * (_align16(len(d)) - len(d))
    return packed, scales
