"""Seeded synthetic inputs shaped like Whisper's Linear layers.

This module holds only input generation (no quantisation and no arithmetic of
the method): the same bytes feed the CUDA path and the CPU oracle.

Generator
---------
A counter-based stream: value i of stream (seed, s) is the splitmix64
finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", 2014) applied to base + (i + 1) * 0x9E3779B97F4A7C15, where
base = finaliser(seed * 0x9E3779B97F4A7C15 + s).  Uniforms are
((v >> 11) + 1) * 2^-53 in (0, 1]; normals come from Box-Muller in fp64 on
consecutive pairs, then are scaled, rounded to fp32, and (for activations and
biases) rounded to bf16 by torch's round-to-nearest-even cast.

Shapes (trained weights and audio are not used: these stand in for them)
------------------------------------------------------------------------
whisper-tiny: d_model 384, FFN 1536.  whisper-large-v3-turbo: d_model 1280
(model card "whisper-large-v3-turbo -- NVFP4", "Honest summary"), FFN 5120,
32 encoder layers x 6 Linears and 4 decoder layers x 10 Linears ("Why the
encoder/decoder split matters"), 1500 encoder frames per 30 s window.
"""

import numpy as np
import torch

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids inside one seed
S_WEIGHT, S_X, S_BIAS, S_OUTLIER = 0, 1, 2, 3


def _mix64(z):
    z = np.asarray(z, np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_next(seed):
    """Successor of a seed in a seed chain (one splitmix64 step)."""
    with np.errstate(over="ignore"):
        s = np.array([int(seed) % (1 << 64)], np.uint64) + GOLDEN
    return int(_mix64(s)[0])


def raw_u64(seed, stream, n, start=0):
    """n raw 64-bit values of stream (seed, stream), from counter start + 1 on (seeds are taken mod 2^64)."""
    with np.errstate(over="ignore"):
        base = _mix64(np.array([int(seed) % (1 << 64)], np.uint64) * GOLDEN + np.uint64(stream))[0]
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(base + ctr * GOLDEN)


def uniform(seed, stream, n):
    v = raw_u64(seed, stream, n)
    return ((v >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed, stream, n, std=1.0, chunk=1 << 24):
    """n samples of N(0, std^2) as float32 (Box-Muller in fp64, in chunks)."""
    out = np.empty(n, np.float32)
    npairs = (n + 1) // 2
    done = 0
    p0 = 0
    while p0 < npairs:
        p1 = min(npairs, p0 + chunk)
        u = raw_u64(seed, stream, 2 * (p1 - p0), start=2 * p0)
        u = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = 2.0 * np.pi * u[1::2]
        z = np.empty(2 * (p1 - p0))
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        take = min(n - done, z.size)
        out[done:done + take] = (z[:take] * std).astype(np.float32)
        done += take
        p0 = p1
    return out


def to_bf16(a_f32):
    """float32 numpy -> torch.bfloat16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a_f32, np.float32)).to(torch.bfloat16)


def bf16_as_f32(t):
    """The exact fp32 values of a bf16 tensor, as numpy."""
    return t.to(torch.float32).numpy()


def weight(seed, N, K, std=0.02):
    return normal(seed, S_WEIGHT, N * K, std).reshape(N, K)


def activations(seed, M, K, std=1.0, outlier_frac=0.0, outlier_mult=20.0):
    """x [M, K] bf16.  With outlier_frac > 0, exactly round(frac * M * K) distinct
    positions, chosen uniformly (the smallest random keys), are multiplied by
    ``outlier_mult`` before the bf16 rounding."""
    x = normal(seed, S_X, M * K, std)
    n_out = int(round(outlier_frac * M * K))
    if n_out:
        keys = raw_u64(seed, S_OUTLIER, M * K)
        pos = np.argpartition(keys, n_out - 1)[:n_out]
        x[pos] = x[pos] * np.float32(outlier_mult)
    return to_bf16(x.reshape(M, K))


def bias(seed, N, std=0.01):
    return to_bf16(normal(seed, S_BIAS, N, std))


# ------------------------------------------------------------------ shapes
TINY = dict(d=384, ffn=1536)
TURBO = dict(d=1280, ffn=5120, enc_layers=32, dec_layers=4, frames=1500)

# decoder layer: self-attn q,k,v,o; cross-attn q,k,v,o; fc1; fc2.  (name, N, K, has_bias)
# Whisper's k projections carry no bias; every other Linear does.
def decoder_layer_linears(d=1280, ffn=5120):
    out = []
    for blk in ("self", "cross"):
        for p in ("q", "k", "v", "o"):
            out.append((f"{blk}_{p}", d, d, p != "k"))
    out.append(("fc1", ffn, d, True))
    out.append(("fc2", d, ffn, True))
    return out


def encoder_layer_linears(d=1280, ffn=5120):
    out = [(f"self_{p}", d, d, p != "k") for p in ("q", "k", "v", "o")]
    out.append(("fc1", ffn, d, True))
    out.append(("fc2", d, ffn, True))
    return out


def encoder_shapes(d=1280, ffn=5120):
    """The three distinct encoder Linear shapes (N, K): q/k/v/o, fc1, fc2."""
    return [("qkvo", d, d), ("fc1", ffn, d), ("fc2", d, ffn)]


def tiny_linears():
    """whisper-tiny fc1 [1536, 384] and its transpose fc2 [384, 1536], both with bias."""
    return [("fc1", TINY["ffn"], TINY["d"], True), ("fc2", TINY["d"], TINY["ffn"], True)]


def turbo_decoder_sweep():
    """40 decoder Linears in model order with their seeds (seed = layer * 16 + index)."""
    out = []
    for layer in range(TURBO["dec_layers"]):
        for i, (name, N, K, hb) in enumerate(decoder_layer_linears()):
            out.append(dict(layer=layer, name=name, N=N, K=K, bias=hb, seed=layer * 16 + i))
    return out


def turbo_full_sweep(seed0=0):
    """232 Linears in model order (32 encoder layers x 6 at M = 1500 in q8_0, then
    4 decoder layers x 10 at M = 1 in q4_0), seeds chained by splitmix64."""
    out = []
    s = seed0
    for layer in range(TURBO["enc_layers"]):
        for name, N, K, hb in encoder_layer_linears():
            out.append(dict(part="encoder", layer=layer, name=name, N=N, K=K, M=TURBO["frames"],
                            fmt="q8_0", bias=hb, seed=s))
            s = splitmix64_next(s)
    for layer in range(TURBO["dec_layers"]):
        for name, N, K, hb in decoder_layer_linears():
            out.append(dict(part="decoder", layer=layer, name=name, N=N, K=K, M=1,
                            fmt="q4_0", bias=hb, seed=s))
            s = splitmix64_next(s)
    return out
