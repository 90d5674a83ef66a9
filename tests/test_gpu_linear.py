"""Fused dequant-matmul (tensor-core and CUDA-core paths) against the fp64 oracle.

Tolerances (stated by the acceptance bar of the method): relative L2 <= 5e-3 on
the bf16 output, max |y - y_ref| <= 1e-2 rms(y_ref) on the fp32-output mode.
Guard rows around y catch out-of-bounds writes."""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import linear as L
from oracle import formats as F
from oracle import quant as Q
from tests.gpu_common import (wq, need_gpu, weight_np, oracle_pack, gpu_pack, with_guard, REL_L2_TOL,
                              MAX_ABS_TOL)
from tests.helpers import rel_l2, max_abs_over_rms

pytestmark = pytest.mark.gpu

SENT_BF16 = -12288.0  # exactly representable in bf16


def run_case(fmt, M, N, K, seed=0, has_bias=True, outliers=0.0, force_simt=False, weights_static=False,
             bar=True):
    W = weight_np(seed, N, K)
    x = wl.activations(seed, M, K, outlier_frac=outliers)
    b = wl.bias(seed, N) if has_bias else None
    p_ref = oracle_pack(fmt, W)
    xf = wl.bf16_as_f32(x)
    bf = wl.bf16_as_f32(b) if has_bias else None
    if fmt == "nvfp4_w4a4":
        y_ref = L.linear_w4a4(xf, p_ref, bf)
    else:
        y_ref = L.linear_w4a16(xf, p_ref, bf)
    packed, scales = gpu_pack(fmt, W)
    xg = x.cuda()
    bg = b.cuda() if has_bias else None
    xin = wq().quant_act_nvfp4(xg) if fmt == "nvfp4_w4a4" else xg
    full16, y16 = with_guard((M, N), torch.bfloat16, SENT_BF16)
    full32, y32 = with_guard((M, N), torch.float32, float("nan"))
    wq().linear_into(y16, xin, packed, scales, fmt, N, K, bg, force_simt=force_simt, weights_static=weights_static)
    wq().linear_into(y32, xin, packed, scales, fmt, N, K, bg, out_f32=True, force_simt=force_simt)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    g16 = full16.float().cpu().numpy()
    g32 = full32.cpu().numpy()
    assert np.all(g16[0] == SENT_BF16) and np.all(g16[-1] == SENT_BF16), "write outside y (bf16)"
    assert np.all(np.isnan(g32[0])) and np.all(np.isnan(g32[-1])), "write outside y (fp32)"
    y16n, y32n = g16[1:-1], g32[1:-1]
    assert np.all(np.isfinite(y32n))
    assert rel_l2(y16n, y_ref) <= REL_L2_TOL, rel_l2(y16n, y_ref)
    if bar:
        assert max_abs_over_rms(y32n, y_ref) <= MAX_ABS_TOL, max_abs_over_rms(y32n, y_ref)
    else:
        # provable elementwise bound for a bf16-rounded weight operand (relative error <= 2^-9 per
        # weight) with fp32 accumulation over K and two fp32 roundings in the epilogue
        w_hat = Q.DEQUANT["nvfp4" if fmt == "nvfp4_w4a4" else fmt](p_ref).astype(np.float64)
        mag = np.abs(xf.astype(np.float64)) @ np.abs(w_hat).T
        bound = (2.0 ** -9 + K * 2.0 ** -23) * mag + 2.0 ** -22 * np.abs(y_ref) + 1e-6
        assert np.all(np.abs(y32n - y_ref) <= bound), float(np.max(np.abs(y32n - y_ref) / bound))
    # the bf16 output is the fp32 output rounded once (same kernel, final cast)
    assert np.array_equal(torch.from_numpy(y32n).to(torch.bfloat16).float().numpy(), y16n)
    return y32n, y_ref


FMTS = ["nf4", "nvfp4", "q4_0", "q8_0"]
NEW_FMTS = ["q4_1", "q5_0", "fp8"]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [
    (1, 1536, 384), (1, 384, 1536),                      # whisper-tiny fc1 / fc2 (decode)
    (1, 1280, 1280), (4, 5120, 1280), (16, 1280, 5120),  # turbo decoder shapes, M in {1, 4, 16}
    (3, 200, 320),                                       # ragged N and K
])
def test_decode_path(fmt, M, N, K):
    need_gpu()
    run_case(fmt, M, N, K, seed=N + K + M)


GEMM_SHAPES = [
    (1500, 1280, 1280),                 # one 30 s window, q/k/v/o
    (300, 5120, 1280),                  # fc1 shape, ragged M
    (37, 1280, 5120),                   # fc2 shape, M between the decode and GEMM tiles
    (130, 200, 256),                    # ragged everything
    (600, 640, 5120),                   # fc2's K with many activation tiles (the longest-K configuration)
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_path(fmt, M, N, K):
    """The acceptance bar on each format's own workload distribution: NVFP4 encoder inputs carry
    0.1 % outliers x20; the q8_0 encoder (and NF4 / q4_0) inputs are plain N(0, 1)."""
    need_gpu()
    run_case(fmt, M, N, K, seed=M + N + K, outliers=0.001 if fmt == "nvfp4" else 0.0)


@pytest.mark.parametrize("fmt", ["nf4", "q4_0", "q8_0"])
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES[:2])
def test_gemm_path_outlier_stress(fmt, M, N, K):
    """Outlier activations on the formats whose decoded weights are not exact in bf16: relative L2
    still within the bar, and every element within the provable bf16-operand error bound."""
    need_gpu()
    run_case(fmt, M, N, K, seed=M + N + K + 1, outliers=0.001, bar=False)


@pytest.mark.parametrize("fmt", FMTS)
def test_simt_path_matches_oracle(fmt):
    need_gpu()
    run_case(fmt, 5, 384, 1536, seed=3, force_simt=True)
    run_case(fmt, 33, 256, 320, seed=4, force_simt=True)


@pytest.mark.parametrize("M,N,K", [(1, 1280, 1280), (16, 5120, 1280), (1500, 1280, 1280), (300, 1280, 5120),
                                   (1100, 200, 768), (1030, 264, 1024), (2048, 128, 256)])
def test_w4a4(M, N, K):
    """Decode sizes (CUDA cores) and the FP4 tensor-core GEMM: ragged activation and weight tiles,
    256- and 512-element chunks, a single chunk."""
    need_gpu()
    run_case("nvfp4_w4a4", M, N, K, seed=100 + M, outliers=0.001)


def test_no_bias_and_static_weights_flag():
    need_gpu()
    run_case("nf4", 16, 1280, 1280, seed=9, has_bias=False, weights_static=True)
    run_case("q4_0", 1, 5120, 1280, seed=10, has_bias=True, weights_static=True)


def test_m_zero_is_noop():
    need_gpu()
    W = weight_np(0, 128, 128)
    packed, scales = gpu_pack("nf4", W)
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    wq().linear_into(y, x, packed, scales, "nf4", 128, 128)
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,K", [(128, 256), (300, 512), (200, 1280), (1280, 512), (1100, 1280)])
def test_w4a4_tensor_path_is_exact_products(M, K):
    """W4A4 on the block-scaled FP4 tensor cores: every product e2m1 * e4m3 * e2m1 * e4m3 is exact
    in fp32, so the fp32 output differs from the fp64 oracle only by the accumulation order and the
    two epilogue roundings: |err| <= (K * 2^-24 + 2^-22) * sum |x_hat| |w_hat|."""
    need_gpu()
    N = 256
    W = weight_np(77 + K, N, K)
    x = wl.activations(77 + M, M, K, outlier_frac=0.001)
    p_ref = oracle_pack("nvfp4", W)
    xf = wl.bf16_as_f32(x)
    a = Q.quant_act_nvfp4(xf)
    x_hat = Q.nvfp4_dequant_parts(a["codes"], a["scales"], a["g"]).astype(np.float64)
    w_hat = Q.nvfp4_dequant(p_ref).astype(np.float64)
    y_ref = x_hat @ w_hat.T
    packed, scales = gpu_pack("nvfp4", W)
    y = wq().linear(wq().quant_act_nvfp4(x.cuda()), packed, scales, "nvfp4_w4a4", N, K, out_f32=True)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    bound = (K * 2.0 ** -24 + 2.0 ** -22) * (np.abs(x_hat) @ np.abs(w_hat).T) + 1e-30
    assert np.all(np.abs(got - y_ref) <= bound), float(np.max(np.abs(got - y_ref) / bound))


@pytest.mark.parametrize("fmt", NEW_FMTS)
@pytest.mark.parametrize("M,N,K", [(1, 1280, 1280), (4, 5120, 1280), (16, 1280, 5120), (3, 200, 384),
                                   (300, 1280, 1280), (37, 640, 5120)])
def test_other_block_types(fmt, M, N, K):
    """q4_1, q5_0 (the other GGUF block types) and FP8 E4M3 weights, decode and encoder sizes."""
    need_gpu()
    run_case(fmt, M, N, K, seed=7 * M + N + K)


@pytest.mark.parametrize("path", ["gemv", "grouped_decode", "gemm"])
def test_fp8_every_code_exact_through_each_path(path):
    """Every finite E4M3 code (both signs, subnormals included) as a weight, picked out by one-hot
    activation rows: with a row scale of 1 each output is exactly the decoded weight, so every
    decode (the CUDA-core GEMV, the tensor-core decode and GEMM tiles) must reproduce the oracle's
    decoded value bit for bit."""
    need_gpu()
    vals = F.e4m3_decode(np.arange(0x7F)).astype(np.float32)          # 0x00 .. 0x7E
    row = np.concatenate([vals, -vals, np.zeros(2, np.float32)])      # 256 values, amax 448
    N, K = 256, 256
    W = np.stack([np.roll(row, n) for n in range(N)]).astype(np.float32)
    p_ref = oracle_pack("fp8", W)
    w_hat = Q.DEQUANT["fp8"](p_ref)
    M = 300 if path == "gemm" else 16
    ks = (np.arange(M) * 37) % K
    x = np.zeros((M, K), np.float32)
    x[np.arange(M), ks] = 1.0
    xb = wl.to_bf16(x).cuda()
    packed, scales = gpu_pack("fp8", W)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    if path == "grouped_decode":
        wq().linear_grouped([(y, xb, packed, scales, N, K, None)], "fp8", out_f32=True)
    else:
        wq().linear_into(y, xb, packed, scales, "fp8", N, K, None, out_f32=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    want = w_hat[:, ks].T.astype(np.float32)
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, want.view(np.uint32) & 0x7FFFFFFF) and \
        np.array_equal(got, want)


# (path, M): one activation row (CUDA-core GEMV), 16 rows grouped (tensor-core decode), 300 rows
# (persistent GEMM), 1500 and 2600 rows (the W4A16 kernel's 128- and 256-row tiles at N = 2048)
NVFP4_CODE_PATHS = [("gemv", 1), ("grouped_decode", 16), ("gemm", 300), ("gemm", 1500), ("gemm", 2600)]


@pytest.mark.parametrize("path,M", NVFP4_CODE_PATHS)
def test_nvfp4_every_code_and_scale_exact_through_each_path(path, M):
    """Every E2M1 code (both signs) under every finite E4M3 block scale (0x01 .. 0x7E, the subnormal
    scales included, plus zero blocks) with g = 1: block b of a row holds the eight E2M1 magnitudes
    and their negatives times S_b = e4m3(b + 1), and the block holding 6 * 448 = 2688 sets g = 1, so
    the packed scale codes are exactly b + 1 and each decoded weight is exactly e2m1 * S_b.  One-hot
    activation rows pick single weights: every output must equal the oracle's decoded weight bit
    for bit on every decode route."""
    need_gpu()
    mags = F.E2M1_MAGNITUDES.astype(np.float32)
    S = F.e4m3_decode(np.arange(1, 0x7F)).astype(np.float32)          # 126 finite positive scales
    blocks = np.concatenate([mags, -mags])[None, :] * S[:, None]       # [126, 16]
    K, N = 2048, 2048
    row = np.zeros(K, np.float32)
    row[:blocks.size] = blocks.reshape(-1)                             # two zero blocks at the end
    W = np.stack([np.roll(row, 16 * n) for n in range(N)]).astype(np.float32)
    p_ref = oracle_pack("nvfp4", W)
    assert p_ref["g"] == np.float32(1)
    assert np.array_equal(p_ref["scales"].reshape(N, K // 16)[0, :126], np.arange(1, 0x7F))
    w_hat = Q.nvfp4_dequant(p_ref)
    ks = (np.arange(M) * 37) % K
    x = np.zeros((M, K), np.float32)
    x[np.arange(M), ks] = 1.0
    xb = wl.to_bf16(x).cuda()
    packed, scales = gpu_pack("nvfp4", W)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    if path == "grouped_decode":
        wq().linear_grouped([(y, xb, packed, scales, N, K, None)], "nvfp4", out_f32=True)
    else:
        wq().linear_into(y, xb, packed, scales, "nvfp4", N, K, None, out_f32=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    want = w_hat[:, ks].T.astype(np.float32)
    got = y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32) & 0x7FFFFFFF, want.view(np.uint32) & 0x7FFFFFFF) and \
        np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(300, 1280, 1280), (1500, 5120, 1280), (130, 1280, 5120)])
def test_w4a4_static_weights_flag(M, N, K):
    """W4A4 launched with programmatic dependent launch right after the activation quantiser: its
    weight tiles stream before the quantiser finishes; the result is the same."""
    need_gpu()
    run_case("nvfp4_w4a4", M, N, K, seed=200 + M, outliers=0.001, weights_static=True)


WIDE_W4A16 = [(2600, 4000, 320), (1100, 20000, 64), (5000, 2000, 1024), (2600, 20000, 128)]
# fewer 256-row tiles than SMs: the same kernel with 128-row activation tiles (fc2 at one window;
# ragged M and N with three chunks; one chunk)
W4A16_128 = [(1500, 1280, 5120), (1000, 1480, 192), (777, 2000, 64)]


@pytest.mark.parametrize("M,N,K", WIDE_W4A16 + W4A16_128)
def test_w4a16_wide_tiles(M, N, K):
    """NVFP4 W4A16 GEMMs on the kernel that decodes each weight tile into shared memory and
    double-buffers its 256- or 128-row accumulators in TMEM: ragged M and N, one to eighty 64-element
    chunks; guard rows, tolerance, and bf16 output = fp32 output rounded once."""
    need_gpu()
    run_case("nvfp4", M, N, K, seed=M + N + K)


@pytest.mark.parametrize("M,N,K", WIDE_W4A16 + W4A16_128)
def test_w4a16_wide_tiles_exact_products(M, N, K):
    """e2m1 * e4m3 weights are exact in bf16 and bf16 * bf16 products exact in fp32, so the fp32
    output differs from the fp64 oracle only by the accumulation order, the global-scale product and
    the bias addition: |err| <= (K + 8) 2^-24 sum |x| |w_hat| + 2^-22 |y|."""
    need_gpu()
    W = weight_np(5 + K, N, K)
    x = wl.activations(5 + M, M, K)
    b = wl.bias(5 + N, N)
    p_ref = oracle_pack("nvfp4", W)
    xf = wl.bf16_as_f32(x).astype(np.float64)
    w_hat = Q.nvfp4_dequant(p_ref).astype(np.float64)
    y_ref = xf @ w_hat.T + wl.bf16_as_f32(b).astype(np.float64)
    packed, scales = gpu_pack("nvfp4", W)
    y = wq().linear(x.cuda(), packed, scales, "nvfp4", N, K, b.cuda(), out_f32=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    got = y.cpu().numpy().astype(np.float64)
    bound = (K + 8) * 2.0 ** -24 * (np.abs(xf) @ np.abs(w_hat).T) + 2.0 ** -22 * np.abs(y_ref) + 1e-30
    assert np.all(np.abs(got - y_ref) <= bound), float(np.max(np.abs(got - y_ref) / bound))
