"""wq_linear_grouped: several independent Linears in one persistent launch, each checked
against the oracle exactly like a single wq_linear call."""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import linear as L
from tests.gpu_common import wq, need_gpu, weight_np, oracle_pack, gpu_pack, REL_L2_TOL, MAX_ABS_TOL
from tests.helpers import rel_l2, max_abs_over_rms

pytestmark = pytest.mark.gpu


def run_group(fmt, specs, out_f32):
    probs, refs, outs = [], [], []
    for i, (M, N, K, has_bias) in enumerate(specs):
        seed = 1000 + 17 * i + M
        W = weight_np(seed, N, K)
        x = wl.activations(seed, M, K, outlier_frac=0.001 if fmt == "nvfp4" else 0.0)
        b = wl.bias(seed, N) if has_bias else None
        refs.append(L.linear_w4a16(wl.bf16_as_f32(x), oracle_pack(fmt, W), wl.bf16_as_f32(b) if has_bias else None))
        packed, scales = gpu_pack(fmt, W)
        full = torch.full((M + 2, N), float("nan"), dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device="cuda")
        outs.append(full)
        probs.append((full[1:M + 1], x.cuda(), packed, scales, N, K, b.cuda() if has_bias else None))
    wq().linear_grouped(probs, fmt, out_f32=out_f32, weights_static=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    for full, ref in zip(outs, refs):
        g = full.float().cpu().numpy()
        assert np.all(np.isnan(g[0])) and np.all(np.isnan(g[-1])), "write outside y"
        y = g[1:-1]
        if out_f32:
            assert max_abs_over_rms(y, ref) <= MAX_ABS_TOL
        else:
            assert rel_l2(y, ref) <= REL_L2_TOL


DECODE_GROUP = [(1, 1280, 1280, True), (1, 1280, 1280, False), (1, 5120, 1280, True), (1, 1280, 5120, True),
                (1, 200, 320, True), (1, 384, 1536, True)]


@pytest.mark.parametrize("fmt", ["nf4", "nvfp4", "q4_0", "q8_0"])
@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("out_f32", [False, True])
def test_grouped_decode(fmt, M, out_f32):
    need_gpu()
    run_group(fmt, [(M, N, K, b) for (_, N, K, b) in DECODE_GROUP], out_f32)


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_grouped_gemm(fmt):
    need_gpu()
    run_group(fmt, [(300, 1280, 1280, True), (130, 5120, 1280, True), (17, 200, 256, False)], out_f32=True)


def test_grouped_full_decoder_layer_set():
    """All 40 decoder Linears of the sweep at M = 1 in one launch (within WQ_GROUP_MAX)."""
    need_gpu()
    specs = [(1, l["N"], l["K"], l["bias"]) for l in wl.turbo_decoder_sweep()]
    run_group("nf4", specs, out_f32=False)


def test_grouped_argument_checks():
    need_gpu()
    import ctypes
    L_ = wq().lib
    assert L_.wq_linear_grouped(None, 1, wq().WQ_NF4, 0, None) == wq().WQ_ERR_ARG
    arr = (wq().wq_problem * 1)()
    assert L_.wq_linear_grouped(ctypes.cast(arr, ctypes.c_void_p), 0, wq().WQ_NF4, 0, None) == wq().WQ_ERR_ARG
    assert L_.wq_linear_grouped(ctypes.cast(arr, ctypes.c_void_p), 49, wq().WQ_NF4, 0, None) == wq().WQ_ERR_ARG
    assert L_.wq_linear_grouped(ctypes.cast(arr, ctypes.c_void_p), 1, wq().WQ_NVFP4_W4A4, 0, None) == wq().WQ_ERR_FMT
