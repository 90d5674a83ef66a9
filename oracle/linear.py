"""The reference contraction of the quantised Linear (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The method replaces an ordinary Linear's matmul by a product with the decoded
weights (PR "asr: add a 4-bit nf4 option for the Whisper engine", "Why NF4 and
not the NVFP4 snapshot": the fused kernel multiplies by the dequantised weights
instead of materialising them).  Its result has a plain definition, written out
here in fp64:

    y[m, n] = sum_k x_hat[m, k] * w_hat[n, k]  (+ bias[n])

W4A16: x_hat = the bf16 activations as given, w_hat = the fp32 decode.
W4A4:  x_hat = the fp32 decode of the oracle's own activation quantisation
       (model card "whisper-large-v3-turbo -- NVFP4", "What is quantized").
"""

import numpy as np

from . import quant as Q


def linear_fp64(x_hat, w_hat, bias=None):
    """fp64 y = x_hat . w_hat^T + bias; x_hat [M, K], w_hat [N, K], bias [N] or None."""
    x = np.asarray(x_hat, np.float64)
    w = np.asarray(w_hat, np.float64)
    y = x @ w.T
    if bias is not None:
        y = y + np.asarray(bias, np.float64)[None, :]
    return y


def linear_w4a16(x_f32, packed, bias=None):
    """W4A16 / W8A16 reference: bf16 activations (given as their fp32 values) times
    the decoded weights of an oracle pack dict."""
    return linear_fp64(x_f32, Q.DEQUANT[packed["fmt"]](packed), bias)


def linear_w4a4(x_f32, packed_nvfp4, bias=None, g_in=None):
    """W4A4 reference: the activations go through the NVFP4 runtime quantiser first."""
    a = Q.quant_act_nvfp4(x_f32, g_in)
    x_hat = Q.nvfp4_dequant_parts(a["codes"], a["scales"], a["g"])
    return linear_fp64(x_hat, Q.nvfp4_dequant(packed_nvfp4), bias)


def rows_fp64(x_hat, w_hat, rows, cols, bias=None):
    """y at the sampled (rows[i], cols[i]) positions only, for checks at sizes where
    the full product is too slow: one fp64 dot product per sample."""
    x = np.asarray(x_hat, np.float64)
    w = np.asarray(w_hat, np.float64)
    out = np.einsum("ik,ik->i", x[rows], w[cols])
    if bias is not None:
        out = out + np.asarray(bias, np.float64)[cols]
    return out
