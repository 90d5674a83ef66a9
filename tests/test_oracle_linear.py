"""Pins of the oracle's fp64 contraction: exact rational arithmetic on tiny cases,
special cases (bias only, identity weights) and the operand orientation."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import linear as L
from oracle import quant as Q


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 5), (3, 7, 4), (5, 2, 8), (1, 6, 3)])
def test_linear_vs_exact_rationals(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = rng.standard_normal((M, K)).astype(np.float32)
    w = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    y = L.linear_fp64(x, w, b)
    assert y.shape == (M, N)
    for m in range(M):
        for n in range(N):
            exact = sum((Fraction(float(x[m, k])) * Fraction(float(w[n, k])) for k in range(K)),
                        Fraction(float(b[n])))
            assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_bias_only_and_identity():
    x = np.arange(12, dtype=np.float32).reshape(3, 4)
    b = np.array([1.5, -2.0], np.float32)
    assert np.array_equal(L.linear_fp64(x, np.zeros((2, 4), np.float32), b), np.tile(b, (3, 1)))
    assert np.array_equal(L.linear_fp64(x, np.eye(4, dtype=np.float32)), x)
    # orientation: y = x . w^T, so row n of w selects output column n
    w = np.zeros((2, 4), np.float32)
    w[1, 3] = 1
    assert np.array_equal(L.linear_fp64(x, w)[:, 1], x[:, 3]) and np.all(L.linear_fp64(x, w)[:, 0] == 0)


def test_sampled_rows_match_full_product():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 64)).astype(np.float32)
    w = rng.standard_normal((11, 64)).astype(np.float32)
    b = rng.standard_normal(11).astype(np.float32)
    full = L.linear_fp64(x, w, b)
    r = np.array([0, 8, 3, 4])
    c = np.array([10, 0, 5, 5])
    assert np.allclose(L.rows_fp64(x, w, r, c, b), full[r, c], rtol=0, atol=1e-12)


def test_w4a4_reference_uses_quantised_activations():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 32)).astype(np.float32)
    w = rng.standard_normal((3, 32)).astype(np.float32)
    p = Q.nvfp4_pack(w)
    a = Q.quant_act_nvfp4(x)
    xh = Q.nvfp4_dequant_parts(a["codes"], a["scales"], a["g"])
    assert np.array_equal(L.linear_w4a4(x, p), L.linear_fp64(xh, Q.nvfp4_dequant(p)))
    assert not np.array_equal(L.linear_w4a4(x, p), L.linear_w4a16(x, p))
