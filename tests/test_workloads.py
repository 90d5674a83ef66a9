"""The seeded input generator: deterministic, independent streams, right statistics."""
import numpy as np
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl


def test_deterministic_and_streams_differ():
    a = wl.normal(5, 0, 1000)
    assert np.array_equal(a, wl.normal(5, 0, 1000))
    assert not np.array_equal(a, wl.normal(5, 1, 1000))
    assert not np.array_equal(a, wl.normal(6, 0, 1000))
    # chunked generation gives the same stream as one chunk
    assert np.array_equal(wl.normal(7, 0, 999, chunk=100), wl.normal(7, 0, 999))


def test_statistics():
    w = wl.weight(0, 512, 512)
    assert abs(float(w.std()) - 0.02) < 0.0005 and abs(float(w.mean())) < 0.0005
    u = wl.uniform(1, 0, 100000)
    assert u.min() > 0 and u.max() <= 1 and abs(u.mean() - 0.5) < 0.01


def test_outliers_exact_count():
    M, K = 300, 256
    x = wl.activations(100, M, K, outlier_frac=0.001)
    base = wl.activations(100, M, K)
    assert x.dtype == torch.bfloat16
    changed = (x != base).sum().item()
    assert changed <= round(0.001 * M * K) and changed >= round(0.001 * M * K) - 2


def test_sweeps():
    dec = wl.turbo_decoder_sweep()
    assert len(dec) == 40 and dec[17]["seed"] == 1 * 16 + 7
    full = wl.turbo_full_sweep()
    assert len(full) == 232
    enc_params = sum(l["N"] * l["K"] for l in full if l["part"] == "encoder")
    dec_params = sum(l["N"] * l["K"] for l in full if l["part"] == "decoder")
    # the model card's "192 Linear, ~630M params" and "40 Linear, ~105M"
    assert enc_params == 629_145_600 and dec_params == 104_857_600
    seeds = [l["seed"] for l in full]
    assert len(set(seeds)) == 232 and seeds[1] == wl.splitmix64_next(seeds[0])
