"""NVFP4 runtime activation quantiser against the oracle: bit-exact codes, scales and g."""
import functools

import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import quant as Q
from tests.gpu_common import wq, need_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,seed", [(1, 1280, 100), (37, 384, 1), (1500, 1280, 100), (1500, 5120, 102),
                                      (6000, 1280, 101), (3, 32, 7)])
@pytest.mark.parametrize("static_g", [False, True])
def test_act_quant_bit_exact(M, K, seed, static_g):
    need_gpu()
    x = wl.activations(seed, M, K, outlier_frac=0.001)
    xf = wl.bf16_as_f32(x)
    g_in = np.float32(0.0031) if static_g else None
    ref = Q.quant_act_nvfp4(xf, g_in)
    gt = torch.tensor([g_in], dtype=torch.float32, device="cuda") if static_g else None
    codes, scales, g = wq().quant_act_nvfp4(x.cuda(), g_in=gt)
    torch.cuda.synchronize()
    assert g.item() == float(ref["g"])
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy().reshape(-1), Q.pack_nibbles(ref["codes"]))


def test_act_quant_all_zero():
    need_gpu()
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    codes, scales, g = wq().quant_act_nvfp4(x)
    assert g.item() == 1.0 and int(codes.sum()) == 0 and int(scales.sum()) == 0


def test_act_quant_many_scales_and_extremes():
    """Blocks spread over a wide range of scales (x spanning 2^-40 .. 2^40 across blocks) with a
    static g that puts some block scales at the bottom of E4M3 and saturates others, every sign of
    zero, and values that make x / S overflow: codes, scales and g bit-exact with the oracle."""
    need_gpu()
    rng = np.random.default_rng(5)
    M, K = 64, 1024
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-40, 40, size=(M, K // 16))).astype(np.float32).repeat(16, axis=1)
    x[0, :16] = -0.0
    x[1, :16] = 0.0
    x[2, 3] = 3.0e38
    x[3, :16] = -1e-30
    xb = wl.to_bf16(x)
    xf = wl.bf16_as_f32(xb)
    for g_in in (np.float32(1e-3), np.float32(7.5), None):
        ref = Q.quant_act_nvfp4(xf, g_in)
        gt = None if g_in is None else torch.tensor([g_in], dtype=torch.float32, device="cuda")
        codes, scales, g = wq().quant_act_nvfp4(xb.cuda(), g_in=gt)
        torch.cuda.synchronize()
        assert g.item() == float(ref["g"])
        assert np.array_equal(scales.cpu().numpy(), ref["scales"])
        assert np.array_equal(codes.cpu().numpy().reshape(-1), Q.pack_nibbles(ref["codes"]))


@pytest.mark.parametrize("static_g", [False, True])
def test_act_quant_many_chunks_ragged(static_g):
    """20.5 M values (16001 x 1280, 1,280,080 blocks: many waves of the quantiser's grid, the last
    one partial, and a grid-stride amax pass of several rounds); bit-exact everywhere."""
    need_gpu()
    M, K = 16001, 1280
    x = wl.activations(103, M, K, outlier_frac=0.001)
    xf = wl.bf16_as_f32(x)
    g_in = np.float32(0.0029) if static_g else None
    ref = Q.quant_act_nvfp4(xf, g_in)
    gt = torch.tensor([g_in], dtype=torch.float32, device="cuda") if static_g else None
    codes, scales, g = wq().quant_act_nvfp4(x.cuda(), g_in=gt)
    torch.cuda.synchronize()
    assert g.item() == float(ref["g"])
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy().reshape(-1), Q.pack_nibbles(ref["codes"]))


@functools.lru_cache(maxsize=1)
def _fc2_b16_activations():
    x = wl.activations(102, 24000, 5120, outlier_frac=0.001)
    return x, wl.bf16_as_f32(x)


@pytest.mark.parametrize("static_g", [False, True])
def test_act_quant_full_fc2_b16_sampled_rows(static_g):
    """The largest encoder activation (M = 24000, K = 5120, 245 MB of bf16): g from the whole
    tensor's amax, codes and scales bit-exact on sampled rows (first and last included)."""
    need_gpu()
    M, K = 24000, 5120
    x, xf = _fc2_b16_activations()
    g_in = np.float32(0.0031) if static_g else None
    gt = torch.tensor([g_in], dtype=torch.float32, device="cuda") if static_g else None
    codes, scales, g = wq().quant_act_nvfp4(x.cuda(), g_in=gt)
    torch.cuda.synchronize()
    g_ref = g_in if static_g else Q.nvfp4_global(np.max(np.abs(xf)))
    assert g.item() == float(g_ref)
    rows = np.concatenate([[0, 1, M // 2, M - 2, M - 1], np.random.default_rng(9).integers(0, M, 59)])
    rc, rs, _ = Q.nvfp4_quantize(xf[rows], g_ref)
    assert np.array_equal(scales.cpu().numpy()[rows], rs)
    assert np.array_equal(codes.cpu().numpy()[rows].reshape(-1), Q.pack_nibbles(rc))
