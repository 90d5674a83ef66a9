"""Fused Q/K/V decode into a KV-cache slab, and a merged cross-attention K|V weight (PR "Run
quantized Whisper on the fused Metal decode path", "Summary": one fused Q/K/V launch, bias applied
on the device, K and V written straight into their slab rows; "Test plan": no copies per token).

Every output is compared with the fp64 oracle, and the slab rows and padding columns around the
written ones must keep their sentinel values."""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import linear as L
from tests.gpu_common import wq, need_gpu, weight_np, oracle_pack, gpu_pack, REL_L2_TOL, MAX_ABS_TOL
from tests.helpers import rel_l2, max_abs_over_rms

pytestmark = pytest.mark.gpu

SENT = -12288.0  # exactly representable in bf16


def _slab(rows, ld, dtype):
    return torch.full((rows, ld), SENT, dtype=dtype, device="cuda")


def _check_slab(slab, t, M, ncols, ref, out_f32):
    """Rows [t, t + M) columns [0, ncols) hold the result; everything else keeps the sentinel."""
    g = slab.float().cpu().numpy()
    got = g[t:t + M, :ncols]
    keep = np.ones_like(g, dtype=bool)
    keep[t:t + M, :ncols] = False
    assert np.all(g[keep] == SENT), "a write outside the addressed slab rows / columns"
    if out_f32:
        assert max_abs_over_rms(got, ref) <= MAX_ABS_TOL
    else:
        assert rel_l2(got, ref) <= REL_L2_TOL


def _qkv_weights(fmt, d, seed):
    Ws = [weight_np(seed + i, d, d) for i in range(3)]
    bs = [wl.bias(seed + i, d) for i in range(3)]
    bs[1] = None  # Whisper's k projection has no bias
    return Ws, bs


@pytest.mark.parametrize("fmt", ["nf4", "nvfp4", "q4_0", "q8_0", "q4_1"])
@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("out_f32", [False, True])
def test_fused_qkv_into_slab(fmt, M, out_f32):
    """Three projections of the same token(s) in one launch; K and V land in rows t .. t+M-1 of
    slabs whose row stride is wider than N."""
    need_gpu()
    d, t, rows, ld = 1280, 5, 12, 1280 + 64
    dt = torch.float32 if out_f32 else torch.bfloat16
    Ws, bs = _qkv_weights(fmt, d, 300 + M)
    x = wl.activations(301 + M, M, d)
    xf = wl.bf16_as_f32(x)
    refs = [L.linear_w4a16(xf, oracle_pack(fmt, W), None if b is None else wl.bf16_as_f32(b)) for W, b in zip(Ws, bs)]
    packs = [gpu_pack(fmt, W) for W in Ws]
    q = _slab(M + 2, d, dt)
    ks, vs = _slab(rows, ld, dt), _slab(rows, ld, dt)
    xg = x.cuda()
    probs = []
    for (p, s), b, out in zip(packs, bs, (q[1:M + 1], ks[t:t + M], vs[t:t + M])):
        probs.append((xg, p, s, d, d, None if b is None else b.cuda(), [(out, d)]))
    wq().linear_grouped_ex(probs, fmt, out_f32=out_f32, weights_static=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    _check_slab(q, 1, M, d, refs[0], out_f32)
    _check_slab(ks, t, M, d, refs[1], out_f32)
    _check_slab(vs, t, M, d, refs[2], out_f32)


@pytest.mark.parametrize("fmt", ["nf4", "q8_0"])
def test_merged_qkv_weight_three_destinations(fmt):
    """One [3d, d] weight packed once; its output columns split three ways (Q buffer, K slab row,
    V slab row) in one problem."""
    need_gpu()
    d, t, rows, M = 1280, 2, 6, 1
    Ws, bs = _qkv_weights(fmt, d, 320)
    Wm = np.concatenate(Ws, axis=0)
    bm = torch.cat([bs[0], torch.zeros(d, dtype=torch.bfloat16), bs[2]])
    x = wl.activations(321, M, d)
    ref = L.linear_w4a16(wl.bf16_as_f32(x), oracle_pack(fmt, Wm), wl.bf16_as_f32(bm))
    p, s = gpu_pack(fmt, Wm)
    q = _slab(M + 2, d, torch.bfloat16)
    ks, vs = _slab(rows, d, torch.bfloat16), _slab(rows, d, torch.bfloat16)
    wq().linear_grouped_ex([(x.cuda(), p, s, 3 * d, d, bm.cuda(),
                             [(q[1:2], d), (ks[t:t + 1], d), (vs[t:t + 1], d)])], fmt, weights_static=True)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    _check_slab(q, 1, M, d, ref[:, :d], False)
    _check_slab(ks, t, M, d, ref[:, d:2 * d], False)
    _check_slab(vs, t, M, d, ref[:, 2 * d:], False)


@pytest.mark.parametrize("fmt", ["nvfp4", "q8_0"])
def test_merged_cross_kv_from_encoder_output(fmt):
    """Cross-attention K|V of one 30 s window: the stacked [2d, d] weight times the encoder output
    (M = 1500) in one GEMM, the K half into the K cache and the V half into the V cache."""
    need_gpu()
    d, M = 1280, 1500
    Wk, Wv = weight_np(340, d, d), weight_np(341, d, d)
    Wm = np.concatenate([Wk, Wv], axis=0)
    bv = wl.bias(341, d)
    bm = torch.cat([torch.zeros(d, dtype=torch.bfloat16), bv])
    x = wl.activations(342, M, d, outlier_frac=0.001 if fmt == "nvfp4" else 0.0)
    ref = L.linear_w4a16(wl.bf16_as_f32(x), oracle_pack(fmt, Wm), wl.bf16_as_f32(bm))
    p, s = gpu_pack(fmt, Wm)
    kc = _slab(M + 3, d + 128, torch.bfloat16)
    vc = _slab(M + 3, d + 128, torch.bfloat16)
    wq().linear_grouped_ex([(x.cuda(), p, s, 2 * d, d, bm.cuda(), [(kc[1:M + 1], d), (vc[2:M + 2], d)])], fmt)
    torch.cuda.synchronize()
    assert wq().last_device_status() == 0
    _check_slab(kc, 1, M, d, ref[:, :d], False)
    _check_slab(vc, 2, M, d, ref[:, d:], False)


def test_grouped_ex_argument_checks():
    need_gpu()
    d = 256
    p, s = gpu_pack("nf4", weight_np(1, d, d))
    x = torch.zeros((1, d), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda")
    bad = [
        [(y[0:1], 100), (y[1:2], 156)],          # first destination not a multiple of 16 columns
        [(y[0:1], 128), (y[1:2], 100)],          # columns do not add up to N
        [(y[0:1, 8:], 256)],                     # misaligned start (16 bytes = 8 bf16 ok) -> use 4
    ]
    with pytest.raises(wq().WQError):
        wq().linear_grouped_ex([(x, p, s, d, d, None, bad[0])], "nf4")
    with pytest.raises(wq().WQError):
        wq().linear_grouped_ex([(x, p, s, d, d, None, bad[1])], "nf4")
    with pytest.raises(wq().WQError):
        wq().linear_grouped_ex([(x, p, s, d, d, None, [(y[0:1, 4:], 256)])], "nf4")
    torch.cuda.synchronize()
