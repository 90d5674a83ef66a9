"""The five workload configurations at full size, run the way bench.py runs them (grouped
launches for the decoder sweeps, one GEMM per Linear for the encoder), against the oracle:
every output where the fp64 reference is cheap, sampled outputs (computed one by one)
where it is not.  Tolerances: rel-L2 <= 5e-3 on bf16 outputs; on the sampled outputs the
max |err| <= 1e-2 rms(sampled reference)."""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import linear as L
from oracle import quant as Q
from tests.gpu_common import wq, need_gpu, REL_L2_TOL, MAX_ABS_TOL
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu


def _pack_both(fmt, seed, N, K):
    W = wl.weight(seed, N, K)
    ref = Q.PACK["nvfp4" if fmt == "nvfp4_w4a4" else fmt](W)
    packed, scales = wq().pack("nvfp4" if fmt == "nvfp4_w4a4" else fmt, torch.from_numpy(W).cuda())
    return ref, packed, scales


def _decoder_sweep(fmt, linears, M):
    probs, refs = [], []
    for l in linears:
        ref, packed, scales = _pack_both(fmt, l["seed"], l["N"], l["K"])
        x = wl.activations(l["seed"] * 7 + M, M, l["K"])
        b = wl.bias(l["seed"], l["N"]) if l["bias"] else None
        refs.append(L.linear_w4a16(wl.bf16_as_f32(x), ref, wl.bf16_as_f32(b) if b is not None else None))
        y = torch.empty((M, l["N"]), dtype=torch.bfloat16, device="cuda")
        probs.append((y, x.cuda(), packed, scales, l["N"], l["K"], b.cuda() if b is not None else None))
    wq().linear_grouped(probs, fmt, weights_static=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    for (y, *_), ref in zip(probs, refs):
        assert rel_l2(y.float().cpu().numpy(), ref) <= REL_L2_TOL


def test_config0_whisper_tiny_nf4():
    """whisper-tiny fc1 [1536, 384] and fc2 [384, 1536], NF4, M = 1, seed 0, with bias."""
    need_gpu()
    _decoder_sweep("nf4", [dict(N=N, K=K, bias=True, seed=0) for _, N, K, _ in wl.tiny_linears()], 1)


@pytest.mark.parametrize("M", [1, 4, 16])
def test_config1_turbo_decoder_nf4_sweep(M):
    """All 40 decoder Linears of the large-v3-turbo shape in one grouped launch, every output."""
    need_gpu()
    _decoder_sweep("nf4", wl.turbo_decoder_sweep(), M)


def _sampled_gemm(fmt, seed, M, N, K, outliers, nsamp=4096):
    ref, packed, scales = _pack_both(fmt, seed, N, K)
    x = wl.activations(seed, M, K, outlier_frac=outliers)
    b = wl.bias(seed, N)
    xg = x.cuda()
    xin = wq().quant_act_nvfp4(xg) if fmt == "nvfp4_w4a4" else xg
    y = wq().linear(xin, packed, scales, fmt, N, K, b.cuda())
    y32 = wq().linear(xin, packed, scales, fmt, N, K, b.cuda(), out_f32=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    rng = np.random.default_rng((seed + M) % (2 ** 63))
    rows = rng.integers(0, M, nsamp)
    cols = rng.integers(0, N, nsamp)
    rows[:4] = [0, M - 1, 0, M - 1]
    cols[:4] = [0, 0, N - 1, N - 1]
    xf = wl.bf16_as_f32(x)
    if fmt == "nvfp4_w4a4":
        # the quantiser works per row once the tensor's global g is known: quantise only the sampled rows
        g = Q.nvfp4_global(np.max(np.abs(xf)))
        codes, sc, g = Q.nvfp4_quantize(xf[rows], g)
        x_rows = Q.nvfp4_dequant_parts(codes, sc, g)
        w_hat = Q.nvfp4_dequant(ref)
        want = np.einsum("ik,ik->i", x_rows.astype(np.float64), w_hat.astype(np.float64)[cols]) + \
            wl.bf16_as_f32(b).astype(np.float64)[cols]
    else:
        w_hat = Q.DEQUANT[fmt](ref)
        want = L.rows_fp64(xf, w_hat, rows, cols, wl.bf16_as_f32(b))
    got16 = y.float().cpu().numpy()[rows, cols]
    got32 = y32.cpu().numpy()[rows, cols].astype(np.float64)
    assert rel_l2(got16, want) <= REL_L2_TOL
    rms = np.sqrt(np.mean(want ** 2))
    assert np.max(np.abs(got32 - want)) <= MAX_ABS_TOL * rms


@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("shape", range(3))
def test_config2_encoder_nvfp4_w4a16(B, shape):
    need_gpu()
    name, N, K = wl.encoder_shapes()[shape]
    _sampled_gemm("nvfp4", 100 + shape, 1500 * B, N, K, outliers=0.001)


@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("shape", range(3))
def test_config3_encoder_nvfp4_w4a4(B, shape):
    need_gpu()
    name, N, K = wl.encoder_shapes()[shape]
    _sampled_gemm("nvfp4_w4a4", 100 + shape, 1500 * B, N, K, outliers=0.001)


def test_config4_sweep_decoder_q4_0():
    """The 40 decoder Linears of the 232-Linear sweep in q4_0 at M = 1, seed-chained."""
    need_gpu()
    dec = [l for l in wl.turbo_full_sweep() if l["part"] == "decoder"]
    _decoder_sweep("q4_0", dec, 1)


@pytest.mark.parametrize("layer", [0, 31])
def test_config4_sweep_encoder_layer_q8_0(layer):
    """One encoder layer (6 Linears, M = 1500) of the 232-Linear sweep in q8_0, sampled outputs."""
    need_gpu()
    enc = [l for l in wl.turbo_full_sweep() if l["part"] == "encoder" and l["layer"] == layer]
    assert len(enc) == 6
    for l in enc:
        _sampled_gemm("q8_0", l["seed"], l["M"], l["N"], l["K"], outliers=0.0, nsamp=2048)
