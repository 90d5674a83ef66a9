"""Helpers shared by the GPU parity tests (inputs come from the seeded generator;
expected values only from oracle/)."""
import numpy as np
import pytest
import torch

from bit_weight_quantized_matmul_gb300 import workloads as wl
from oracle import quant as Q

REL_L2_TOL = 5e-3        # relative L2 of the bf16 output against the fp64 oracle
MAX_ABS_TOL = 1e-2       # max |y - y_ref| / rms(y_ref), on the fp32-output mode


def wq():
    from bit_weight_quantized_matmul_gb300 import wq as mod
    return mod


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def weight_np(seed, N, K, std=0.02):
    return wl.weight(seed, N, K, std)


def oracle_pack(fmt, W):
    return Q.PACK["nvfp4" if fmt == "nvfp4_w4a4" else fmt](W)


def gpu_pack(fmt, W_np):
    W = torch.from_numpy(np.ascontiguousarray(W_np)).cuda()
    return wq().pack(fmt, W)


def blob_bytes(t, n):
    return t[:n].cpu().numpy().tobytes()


def with_guard(shape, dtype, fill):
    """A buffer with one guard row before and after; returns (full, view)."""
    M, N = shape
    full = torch.full((M + 2, N), fill, dtype=dtype, device="cuda")
    return full, full[1:M + 1]
