"""Deterministic rounding-edge inputs through the device encoders, bit-exact against the oracle.

Random weights and activations reach the tie branches of the encoders only by chance.  Every
input here is built so that a value lands exactly on a decision point of one encoder (and one
ulp either side of it), so that a comparison written as `>` where `>=` is meant, a tie sent the
wrong way, or a lost sign of zero changes a byte:

* NVFP4 / W4A4 activations (model card "whisper-large-v3-turbo -- NVFP4", "What is quantized"):
  every E2M1 tie x/S in {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} with both signs, tiny negatives
  that round to -0 (code 8), E4M3 block-scale ties, subnormal and underflowing block scales,
  saturating block scales with a static global scale; the hand-worked 2 x 16 NVFP4 matrix.
* q4_0 / q8_0 (PR "Run quantized Whisper on the fused Metal decode path", "Summary"): the
  hand-worked rows, rint half-way cases of both signs, the clamp side of q4_0.
* NF4 (PR "asr: add a 4-bit nf4 option for the Whisper engine", "What's here"): values exactly on
  every fp32 codebook midpoint and one ulp either side, for absmax 1 and a power-of-two absmax.

Expected bytes come from oracle/ only; the fixtures' own values are pinned in the oracle tests.
"""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import formats as F
from oracle import quant as Q
from tests.gpu_common import wq, need_gpu, oracle_pack, gpu_pack, blob_bytes
from tests.helpers import golden_dict

pytestmark = pytest.mark.gpu

E2M1_TIES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)


def _check_pack(fmt, W):
    """GPU pack of W == oracle pack, byte for byte, and the decode export == oracle decode."""
    W = np.ascontiguousarray(W, np.float32)
    N, K = W.shape
    ref = oracle_pack(fmt, W)
    ref_packed, ref_scales = Q.to_blobs(ref)
    packed, scales = gpu_pack(fmt, W)
    torch.cuda.synchronize()
    assert blob_bytes(packed, len(ref_packed)) == ref_packed, f"{fmt}: packed bytes"
    assert blob_bytes(scales, len(ref_scales)) == ref_scales, f"{fmt}: scales bytes"
    deq = wq().dequant(fmt, packed, scales, N, K).cpu().numpy()
    exp = Q.DEQUANT[fmt](ref)
    assert np.array_equal(deq.view(np.uint32), exp.view(np.uint32)), f"{fmt}: decoded values"
    assert wq().last_device_status() == 0
    return ref


def _ulp_neighbours(v):
    v = np.asarray(v, np.float32)
    return np.concatenate([v, np.nextafter(v, np.float32(-np.inf)), np.nextafter(v, np.float32(np.inf))])


# ------------------------------------------------------------------ scalar encoders
def test_scalar_encoders_on_every_decision_point():
    """The library's E2M1 / E4M3 encoders and the hardware cvt.rn.satfinite conversions on ties,
    signed zeros, subnormal E4M3 values and saturation, against the oracle's encoders."""
    need_gpu()
    e4 = F.E4M3_FINITE_POS.astype(np.float32)
    e4_mid = ((F.E4M3_FINITE_POS[:-1] + F.E4M3_FINITE_POS[1:]) / 2).astype(np.float32)
    e2 = F.E2M1_MAGNITUDES.astype(np.float32)
    xs = np.concatenate([
        _ulp_neighbours(E2M1_TIES), -_ulp_neighbours(E2M1_TIES), e2, -e2,
        np.array([0.0, -0.0, 1e-30, -1e-30, -0.1, -0.2499, 6.0, 6.5, 7.0, -7.0, 1e30, -1e30], np.float32),
        _ulp_neighbours(e4_mid), e4, -e4,
        np.array([2.0 ** -10, 3 * 2.0 ** -10, 2.0 ** -11, 448.0, 464.0, 465.0, 1e6], np.float32),
    ]).astype(np.float32)
    out = wq().selftest_encoders(torch.from_numpy(xs).cuda()).cpu().numpy()
    exp_e2m1 = F.e2m1_encode(xs)
    fin = np.abs(xs) < 3e38
    exp_e4m3 = F.e4m3_encode_satfinite(xs)
    assert np.array_equal(out[:, 0], exp_e2m1), xs[out[:, 0] != exp_e2m1]
    assert np.array_equal(out[fin, 2], exp_e4m3[fin]), xs[fin][out[fin, 2] != exp_e4m3[fin]]
    # the hardware conversions round the same way, including -0 for tiny negatives
    assert np.array_equal(out[:, 1], out[:, 0]), xs[out[:, 1] != out[:, 0]]
    assert np.array_equal(out[fin, 3], out[fin, 2]), xs[fin][out[fin, 3] != out[fin, 2]]


# ------------------------------------------------------------------ NVFP4 weights
def test_nvfp4_worked_matrix_on_device():
    """The hand-worked 2 x 16 matrix (ties, saturation, -0, block-scale rounding), zero-padded to
    K = 32 (the packer's row rule); its bytes are also the fixture's."""
    need_gpu()
    g = golden_dict("nvfp4_worked.txt")
    W = np.zeros((2, 32), np.float32)
    W[:, :16] = np.array([[float(v) for v in row] for row in g["x"]], np.float32)
    ref = _check_pack("nvfp4", W)
    codes = ref["codes"].reshape(2, 32)[:, :16].reshape(-1)
    exp_codes = np.array([[int(c) for c in row] for row in g["codes"]], np.uint8).reshape(-1)
    assert np.array_equal(codes, exp_codes)


def _nvfp4_edge_rows():
    """Rows of 16-blocks whose amax_b / 6 (with g = 1: one block holds 2688) hits E4M3 ties,
    the subnormal grid, the underflow tie to zero and the top of the range; the other elements
    of each block land on E2M1 ties relative to the block's decoded scale."""
    amax_over_6 = [17.0,                  # tie 16 / 18 -> 16 (even mantissa)
                   19.0,                  # tie 18 / 20 -> 20
                   1.0625,                # tie 1 / 1.125 -> 1
                   1.5 * 2.0 ** -9,       # subnormal tie 2^-9 / 2^-8 -> 2^-8
                   2.5 * 2.0 ** -9,       # subnormal tie -> 2 * 2^-9
                   2.0 ** -10,            # tie 0 / 2^-9 -> 0: the block scale underflows, codes 0
                   0.75 * 2.0 ** -10,     # below the tie: underflow
                   448.0, 100.0, 0.3]
    rows = []
    for a6 in amax_over_6:
        blk = np.zeros(16, np.float32)
        blk[0] = np.float32(a6 * 6.0)
        S = float(F.e4m3_decode(F.e4m3_encode_satfinite(np.float32(a6))))
        ties = (E2M1_TIES * np.float32(S)).astype(np.float32)
        ties = np.where(ties <= blk[0], ties, np.float32(0))  # stay below the block amax
        blk[1:8] = ties
        blk[8:15] = -ties
        blk[15] = -np.float32(S * 0.1)   # rounds to zero with a negative sign: code 8
        rows.append(blk)
    top = np.zeros(16, np.float32)
    top[0] = 2688.0                       # sets g = 1
    rows.append(top)
    return np.stack(rows).reshape(1, -1)  # one row, K = 16 * 11 = 176 -> pad to 192


def test_nvfp4_pack_scale_ties_and_subnormal_scales():
    need_gpu()
    r = _nvfp4_edge_rows()
    W = np.zeros((3, 192), np.float32)
    W[0, :r.shape[1]] = r[0]
    W[1, :r.shape[1]] = -r[0]
    W[2, 16:32] = r[0, :16] * np.float32(0.5)
    _check_pack("nvfp4", W)


# ------------------------------------------------------------------ NVFP4 activations
def _act_tie_matrix():
    """bf16 activations: per row a set of 16-blocks whose decoded block scale S is a power of two
    and whose other elements sit on every E2M1 tie (both signs), one bf16 ulp either side of a
    tie, and tiny negatives; with g = 1 the block amax 6 * S gives s = E4M3(S) exactly."""
    blocks = []
    for S in (1.0, 0.5, 2.0 ** -6, 2.0 ** -9, 64.0):
        b = np.zeros(16, np.float32)
        b[0] = 6.0 * S
        b[1:8] = E2M1_TIES * S
        b[8:15] = -E2M1_TIES * S
        b[15] = -0.05 * S
        blocks.append(b)
        # ties nudged by one bf16 ulp (bf16 keeps 8 significant bits)
        b2 = np.zeros(16, np.float32)
        b2[0] = 6.0 * S
        up = (E2M1_TIES * (1 + 2.0 ** -7) * S).astype(np.float32)
        dn = (E2M1_TIES * (1 - 2.0 ** -8) * S).astype(np.float32)
        b2[1:8] = up
        b2[8:15] = -dn
        b2[15] = -6.0 * S
        blocks.append(b2)
    sat = np.zeros(16, np.float32)      # amax 6016 -> ratio 1002.67 -> s saturates at 448
    sat[0] = 6016.0
    sat[1] = -3000.0
    sat[2] = 2688.0
    blocks.append(sat)
    zero = np.zeros(16, np.float32)
    zero[3] = -0.0
    blocks.append(zero)
    row = np.concatenate(blocks)                           # 12 blocks = 192
    x = np.stack([row, -row, row[::-1].copy(), np.roll(row, 16)])
    return wl.to_bf16(x)


@pytest.mark.parametrize("g_in", [1.0, 0.5, None])
def test_act_quant_ties_and_signed_zeros(g_in):
    """Static g = 1 puts x / S exactly on the ties; g = 0.5 and the dynamic g move the block scales
    onto other E4M3 values and, for the saturating block, past 448."""
    need_gpu()
    x = _act_tie_matrix()
    xf = wl.bf16_as_f32(x)
    gv = None if g_in is None else np.float32(g_in)
    ref = Q.quant_act_nvfp4(xf, gv)
    gt = None if g_in is None else torch.tensor([g_in], dtype=torch.float32, device="cuda")
    codes, scales, g = wq().quant_act_nvfp4(x.cuda(), g_in=gt)
    torch.cuda.synchronize()
    assert g.item() == float(ref["g"])
    assert np.array_equal(scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(codes.cpu().numpy().reshape(-1), Q.pack_nibbles(ref["codes"]))
    if g_in == 1.0:
        # the fixture really lands on the ties: the oracle's codes for the tie elements of the
        # S = 1 block are the even neighbours, and -0.05 is stored as -0
        c = ref["codes"][0, :16]
        assert list(c[1:8]) == [0, 2, 2, 4, 4, 6, 6] and list(c[8:15]) == [8, 10, 10, 12, 12, 14, 14]
        assert c[15] == 8


# ------------------------------------------------------------------ q4_0 / q8_0
def _gguf_worked(name):
    g = golden_dict(name)
    W = np.zeros((1, 64), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    return W


@pytest.mark.parametrize("fmt,golden", [("q4_0", "q4_0_worked.txt"), ("q8_0", "q8_0_worked.txt")])
def test_gguf_worked_rows_on_device(fmt, golden):
    need_gpu()
    W = _gguf_worked(golden)
    ref = _check_pack(fmt, np.concatenate([W, -W, W * np.float32(0.5)]))
    g = golden_dict(golden)
    assert [int(h, 16) for h in g["d"][0]] == list(ref["d"].view(np.uint16)[:2])


def test_gguf_rint_halfway_cases():
    """Blocks whose d is a power of two so that x / d lands on k + 0.5 for every k in range,
    both signs (rint half to even), plus q4_0's clamp side (+8 steps -> code 15 at the top)."""
    need_gpu()
    # q8_0: amax 127 -> d = 1 exactly; elements k + 0.5
    q8 = np.zeros((4, 64), np.float32)
    q8[:, 0] = 127.0
    q8[0, 1:32] = np.arange(31, dtype=np.float32) + 0.5
    q8[1, 1:32] = -(np.arange(31, dtype=np.float32) + 0.5)
    q8[2, 32] = -127.0
    q8[2, 33:64] = np.arange(95, 126, dtype=np.float32) + 0.5
    q8[3, 32] = 254.0                     # d = 2: x / d = (2k + 1) / 2
    q8[3, 33:64] = 2 * np.arange(31, dtype=np.float32) + 1.0
    _check_pack("q8_0", q8)
    # q4_0: extreme -4 -> d = 0.5; x = (k + 0.5) * 0.5 for k in -8..6
    q4 = np.zeros((3, 64), np.float32)
    q4[:, 0] = -4.0
    halves = ((np.arange(-8, 7, dtype=np.float32) + 0.5) * 0.5).astype(np.float32)
    q4[0, 1:1 + halves.size] = halves
    q4[1, 1:1 + halves.size] = -halves
    q4[2, 32] = 4.0                       # extreme +4 -> d = -0.5: the +side clamps
    q4[2, 33:33 + halves.size] = halves
    q4[2, 60] = -4.0                      # x / d = +8 -> q = 16 -> clamped to 15
    _check_pack("q4_0", q4)


# ------------------------------------------------------------------ NF4
def test_nf4_codebook_midpoints_and_neighbours():
    """Values exactly on every fp32 midpoint of the codebook (ties go to the lower code) and one
    ulp either side, in blocks whose absmax is 1 (v = w exactly) or 2^-5 (exact scaling)."""
    need_gpu()
    cb = F.NF4_CODEBOOK
    mids = ((cb[:-1] + cb[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float32)
    vals = _ulp_neighbours(mids)                           # 45 values
    rows = []
    for a in (1.0, 2.0 ** -5):
        blk = np.zeros(64, np.float32)
        blk[0] = np.float32(a)
        blk[1:1 + vals.size] = (vals * np.float32(a)).astype(np.float32)
        blk[50] = -np.float32(a)                           # the codebook's -1 end
        rows.append(blk)
        neg = blk.copy()
        neg[0] = -np.float32(a)                            # absmax from a negative element
        rows.append(neg)
    W = np.stack(rows)
    W = np.concatenate([W, W * np.float32(0.75)], axis=1)  # K = 128: a second absmax per row
    ref = _check_pack("nf4", W)
    # the fixture's midpoints really are ties: those elements got the lower code
    codes = ref["codes"].reshape(4, 128)
    assert list(codes[0, 1:16]) == list(range(15))


def test_fp8_weight_worked_matrix_and_ties():
    """The hand-worked FP8 matrix (E4M3 ties, subnormals, the tie to zero, -0), and rows whose
    w / s lands exactly on every E4M3 midpoint (s = 1: the row amax is 448)."""
    need_gpu()
    g = golden_dict("fp8_worked.txt")
    W = np.zeros((6, 288), np.float32)
    x0 = [float(v) for v in g["x0"][0]]
    W[0, :len(x0)] = x0
    W[0, 10] = -0.0
    W[1] = W[0] * 2
    x3 = [float(v) for v in g["x3"][0]]
    W[3, :len(x3)] = x3
    mids = ((F.E4M3_FINITE_POS[:-1] + F.E4M3_FINITE_POS[1:]) / 2).astype(np.float32)   # 126 values
    W[4, 0] = 448.0
    W[4, 1:1 + mids.size] = mids
    W[4, 128:128 + mids.size] = -mids
    W[5, 0] = -448.0
    W[5, 1:1 + mids.size] = np.nextafter(mids, np.float32(0))
    W[5, 128:128 + mids.size] = np.nextafter(mids, np.float32(1e9))
    _check_pack("fp8", W)


@pytest.mark.parametrize("golden", ["q4_1_worked.txt", "q5_0_worked.txt"])
def test_other_gguf_worked_rows(golden):
    """The hand-worked q4_1 and q5_0 rows (rint ties both ways, the clamp side, -0 scales of
    all-zero blocks) through the GPU packers."""
    need_gpu()
    g = golden_dict(golden)
    fmt = golden.split("_worked")[0]
    W = np.zeros((1, 128), np.float32)
    if fmt == "q4_1":
        W[0, :32] = float(g["rest0"][0][0])
        W[0, 32:64] = float(g["rest1"][0][0])
    x0 = [float(v) for v in g["x0"][0]]
    x1 = [float(v) for v in g["x1"][0]]
    W[0, :len(x0)] = x0
    W[0, 32:32 + len(x1)] = x1
    _check_pack(fmt, np.concatenate([W, -W, W * np.float32(0.25)]))
