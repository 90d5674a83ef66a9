"""The C-ABI library loads and exports every symbol include/wq.h declares; host-side
argument checks and storage sizes (no GPU needed: every call here fails its checks,
or only computes sizes, before any CUDA call)."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import quant as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")


@pytest.fixture(scope="module")
def wq():
    from bit_weight_quantized_matmul_gb300 import build
    build.build()
    from bit_weight_quantized_matmul_gb300 import wq as mod
    return mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(wq_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["wq_pack_nf4", "wq_pack_nvfp4", "wq_pack_q4_0", "wq_pack_q8_0", "wq_linear", "wq_linear_ex",
              "wq_quant_act_nvfp4", "wq_dequant", "wq_packed_bytes", "wq_scales_bytes"]:
        assert n in names


def test_library_exports_every_declared_symbol(wq):
    lib = ctypes.CDLL(wq.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n


@pytest.mark.parametrize("fmt,N,K", [("nf4", 1536, 384), ("nf4", 3, 6400), ("nf4", 1280, 1280),
                                     ("nvfp4", 1280, 5120), ("nvfp4", 2, 32), ("q4_0", 384, 1536),
                                     ("q8_0", 5120, 1280), ("q8_0", 1, 32), ("q4_1", 3, 128), ("q4_1", 1280, 1280),
                                     ("q5_0", 5, 384), ("q5_0", 1280, 5120), ("fp8", 3, 32), ("fp8", 1280, 1280)])
def test_sizes_match_oracle_blobs(wq, fmt, N, K):
    W = np.random.default_rng(0).standard_normal((N, K)).astype(np.float32) * 0.02
    packed, scales = Q.to_blobs(Q.PACK[fmt](W))
    assert wq.packed_bytes(fmt, N, K) == len(packed)
    assert wq.scales_bytes(fmt, N, K) == len(scales)


def test_size_rules(wq):
    assert wq.packed_bytes("nf4", 4, 96) == 0          # K % 64
    assert wq.packed_bytes("q4_0", 4, 48) == 0         # K % 32
    assert wq.packed_bytes("nvfp4", 4, 48) == 0        # K % 32 (16-blocks, 16-byte rows)
    assert wq.packed_bytes(9, 4, 64) == 0              # unknown format
    assert wq.packed_bytes("q5_0", 4, 64) == 0         # K % 128 (whole storage units)
    assert wq.packed_bytes("q5_0", 4, 256) == 4 * 160 and wq.packed_bytes("fp8", 3, 64) == 192
    assert wq.packed_bytes("nf4", 0, 64) == 0 and wq.scales_bytes("q8_0", 0, 32) == 0


def test_argument_checks_before_any_launch(wq):
    L = wq.lib
    fake = ctypes.c_void_p(0x10000)     # never dereferenced: every call below fails its checks first
    odd = ctypes.c_void_p(0x10008)
    assert L.wq_pack_nf4(fake, 4, 96, fake, fake, None) == wq.WQ_ERR_SHAPE
    assert L.wq_pack_nf4(None, 4, 64, fake, fake, None) == wq.WQ_ERR_ARG
    assert L.wq_pack_q8_0(odd, 4, 64, fake, fake, None) == wq.WQ_ERR_ALIGN
    assert L.wq_pack_nvfp4(fake, -1, 64, fake, fake, None) == wq.WQ_ERR_ARG
    assert L.wq_linear(fake, fake, fake, 9, 1, 4, 64, None, fake, None) == wq.WQ_ERR_FMT
    assert L.wq_linear(fake, fake, fake, wq.WQ_Q5_0, 1, 4, 64, None, fake, None) == wq.WQ_ERR_SHAPE
    assert L.wq_linear(None, fake, fake, wq.WQ_NF4, 1, 4, 64, None, fake, None) == wq.WQ_ERR_ARG
    assert L.wq_linear(fake, fake, fake, wq.WQ_NF4, 1, 4, 96, None, fake, None) == wq.WQ_ERR_SHAPE
    assert L.wq_linear(odd, fake, fake, wq.WQ_NF4, 1, 4, 64, None, fake, None) == wq.WQ_ERR_ALIGN
    assert L.wq_linear(fake, fake, fake, wq.WQ_NF4, 1, 4, 64, odd, fake, None) == wq.WQ_ERR_ALIGN
    assert L.wq_linear(fake, fake, fake, wq.WQ_NF4, -1, 4, 64, None, fake, None) == wq.WQ_ERR_ARG
    assert L.wq_linear(fake, fake, fake, wq.WQ_NF4, 0, 4, 64, None, fake, None) == wq.WQ_OK  # M == 0: no-op
    assert L.wq_linear_ex(fake, fake, fake, wq.WQ_NF4, 1, 4, 64, None, fake, 1 << 9, None) == wq.WQ_ERR_ARG
    assert L.wq_quant_act_nvfp4(fake, 2, 48, None, fake, fake, fake, None) == wq.WQ_ERR_SHAPE
    assert L.wq_quant_act_nvfp4(odd, 2, 64, None, fake, fake, fake, None) == wq.WQ_ERR_ALIGN
    assert L.wq_dequant(fake, fake, 0, 4, 64, fake, None) == wq.WQ_ERR_FMT
    # W4A4: x is a host struct of device pointers; a NULL member is rejected
    act = wq.wq_act_nvfp4(0x10000, None, 0x10000)
    xp = ctypes.cast(ctypes.pointer(act), ctypes.c_void_p)
    assert L.wq_linear(xp, fake, fake, wq.WQ_NVFP4_W4A4, 1, 4, 64, None, fake, None) == wq.WQ_ERR_ARG
    # the failure-path self test checks its poll count before launching
    assert L.wq_selftest_timeout(0, None) == wq.WQ_ERR_ARG
    assert L.wq_selftest_timeout((1 << 20) + 1, None) == wq.WQ_ERR_ARG


def test_status_strings(wq):
    for s in range(-6, 1):
        assert len(wq.lib.wq_status_string(s)) > 0
    assert wq.lib.wq_status_string(-99) == b"unknown status"
