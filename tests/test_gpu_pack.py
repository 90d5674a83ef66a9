"""GPU packers and decode export against the oracle: bit-exact bytes and values."""
import numpy as np
import pytest
import torch

from oracle import quant as Q
from oracle import formats as F
from tests.gpu_common import wq, need_gpu, weight_np, oracle_pack, gpu_pack, blob_bytes

pytestmark = pytest.mark.gpu

SHAPES = [
    (1536, 384), (384, 1536),          # whisper-tiny fc1 / fc2
    (1280, 1280), (5120, 1280), (1280, 5120),   # large-v3-turbo Linears
    (3, 6400),                          # 300 NF4 blocks: a ragged double-quant group
    (1, 64), (7, 128), (200, 320),      # small and ragged
    (1000, 1088),                       # 17000 NF4 blocks: the parallel double-quant with a ragged last group
]


BLOCK = {"nf4": 64, "nvfp4": 32, "q4_0": 32, "q8_0": 32, "q4_1": 128, "q5_0": 128, "fp8": 32}


@pytest.mark.parametrize("fmt", ["nf4", "nvfp4", "q4_0", "q8_0", "q4_1", "q5_0", "fp8"])
@pytest.mark.parametrize("N,K", SHAPES)
def test_pack_and_dequant_bit_exact(fmt, N, K):
    need_gpu()
    if K % BLOCK[fmt]:
        pytest.skip("shape not valid for format")
    W = weight_np(N * 7 + K, N, K)
    W[0, :16] *= 30.0                  # an outlier block
    if N > 2:
        W[2, :64] = 0.0                # an all-zero block
    ref = oracle_pack(fmt, W)
    ref_packed, ref_scales = Q.to_blobs(ref)
    packed, scales = gpu_pack(fmt, W)
    torch.cuda.synchronize()
    assert blob_bytes(packed, len(ref_packed)) == ref_packed
    assert blob_bytes(scales, len(ref_scales)) == ref_scales
    deq = wq().dequant(fmt, packed, scales, N, K).cpu().numpy()
    exp = Q.DEQUANT[fmt](ref)
    assert np.array_equal(deq.view(np.uint32), exp.view(np.uint32))
    assert wq().last_device_status() == 0


def test_nf4_codebook_on_device_equals_oracle():
    """Every NF4 code with absmax decoding to exactly 1.0 returns the kernel's codebook value."""
    need_gpu()
    N, K = 1, 64
    codes = np.arange(64, dtype=np.uint8) % 16
    packed = torch.from_numpy(Q.pack_nibbles(codes)).cuda()
    # absmax code 0, s2 = 0, offset = 1.0  ->  a_hat = 0 * 0 + 1 = 1
    blob = np.zeros(16 + 4 + 4, np.uint8)
    blob[20:24] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    scales = torch.from_numpy(blob).cuda()
    deq = wq().dequant("nf4", packed, scales, N, K).cpu().numpy().reshape(-1)
    assert np.array_equal(deq[:16].view(np.uint32), F.NF4_CODEBOOK.view(np.uint32))


def test_e4m3_e2m1_decoders_exhaustive():
    """All 16 E2M1 codes x all 126 finite positive E4M3 scale bytes through the NVFP4 decoder."""
    need_gpu()
    K = 16 * 128
    codes = np.tile(np.arange(16, dtype=np.uint8), K // 16)
    sf = np.arange(128, dtype=np.uint8)
    sf[127] = 0x7E
    blob = np.zeros(128 + 4, np.uint8)
    blob[:128] = sf
    blob[128:132] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    deq = wq().dequant("nvfp4", torch.from_numpy(Q.pack_nibbles(codes)).cuda(), torch.from_numpy(blob).cuda(),
                       1, K).cpu().numpy().reshape(128, 16)
    exp = (F.e2m1_decode(np.arange(16))[None, :] * F.e4m3_decode(sf)[:, None]).astype(np.float32)
    assert np.array_equal(deq.view(np.uint32), exp.view(np.uint32))


def test_zero_sized_is_noop():
    need_gpu()
    W = torch.zeros((0, 64), device="cuda")
    p, s = wq().pack("nf4", W)
    assert p.numel() >= 0
