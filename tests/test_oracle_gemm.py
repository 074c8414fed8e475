"""Pins for the oracle's GEMMs.

The fp64 NVFP4 GEMM is checked against a second, integer-only evaluation of the
same sum (exact by construction), against one-hot operands whose product is a
closed form, and against sampled-row consistency.  The fp64 BF16 GEMM is checked
against numpy's float64 matmul (a library routine) and one-hot operands.
"""

from fractions import Fraction

import numpy as np
import torch

import workloads


def _nvfp4_operand(rows, K, seed, stream):
    c, sf, s = workloads.random_nvfp4_operand(rows, K, seed, stream)
    return c.numpy(), sf.numpy(), s.numpy()


def test_nvfp4_gemm_matches_integer_evaluation(orc):
    M, N, K = 12, 20, 512
    ac, asf, a_s = _nvfp4_operand(M, K, 0, 0)
    wc, wsf, _ = _nvfp4_operand(N, K, 0, 1)
    w_s = np.float32(0.37)
    y, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, w_s)
    T = orc.gemm_nvfp4_exact(ac, asf, wc, wsf)
    for m in range(M):
        for n in range(N):
            exact = Fraction(float(a_s[m])) * Fraction(float(w_s)) * Fraction(int(T[m, n]), 2 ** 20)
            err = abs(Fraction(y[m, n]) - exact)
            assert err <= Fraction(K) * Fraction(2) ** -52 * Fraction(S[m, n]) + Fraction(2) ** -1000


def test_nvfp4_gemm_one_hot_rows_pick_weight_columns(orc):
    """A rows with a single nonzero element (code 1.0 at k*, scale 1.0) give
    y[m, n] = a_s[m] * w_hat[n, k*]: catches a transposed operand or a wrong
    K index."""
    M, N, K = 4, 8, 128
    wc, wsf, _ = _nvfp4_operand(N, K, 1, 2)
    w_s = np.float32(1.5)
    ks = [0, 17, 64, 127]
    ac = np.zeros((M, K // 2), np.uint8)
    asf = np.full((M, K // 16), 0x38, np.uint8)  # 1.0
    a_s = np.array([1.0, 2.0, 0.5, 4.0], np.float32)
    for m, k in enumerate(ks):
        ac[m, k // 2] = 0x2 << (4 * (k % 2))  # code 0x2 = 1.0
    bias = (np.arange(N, dtype=np.float32) * 0.25).astype(np.float32)
    bias_bits = (bias.view(np.uint32) >> 16).astype(np.uint16)
    y, _ = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, w_s, bias_bits=bias_bits)
    w_hat = orc.dequantize(wc, wsf, np.array([w_s]), "tensor")
    for m, k in enumerate(ks):
        assert np.array_equal(y[m], a_s[m] * w_hat[:, k] + bias)


def test_nvfp4_gemm_sampled_rows_equal_full(orc):
    M, N, K = 9, 5, 64
    ac, asf, a_s = _nvfp4_operand(M, K, 2, 3)
    wc, wsf, _ = _nvfp4_operand(N, K, 2, 4)
    y, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, np.float32(1.0))
    rows = np.array([8, 0, 3])
    y2, S2 = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, np.float32(1.0), rows=rows)
    assert np.array_equal(y[rows], y2) and np.array_equal(S[rows], S2)
    T = orc.gemm_nvfp4_exact(ac, asf, wc, wsf)
    assert np.array_equal(T[rows], orc.gemm_nvfp4_exact(ac, asf, wc, wsf, rows=rows))


def _bits(t):
    return workloads.bf16_bits(t)


def test_bf16_gemm_matches_numpy_float64(orc):
    g = torch.Generator().manual_seed(0)
    M, N, K = 7, 11, 300
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    b = torch.randn(N, generator=g).to(torch.bfloat16)
    y, S = orc.gemm_bf16(_bits(x), _bits(w), _bits(b))
    ref = x.double().numpy() @ w.double().numpy().T + b.double().numpy()
    tol = K * 2.0 ** -52 * S + 2.0 ** -52 * np.abs(ref)
    assert np.all(np.abs(y - ref) <= tol)
    assert np.allclose(S, np.abs(x.double().numpy()) @ np.abs(w.double().numpy()).T, rtol=1e-12)


def test_bf16_gemm_one_hot(orc):
    g = torch.Generator().manual_seed(1)
    N, K = 6, 40
    w = torch.randn(N, K, generator=g).to(torch.bfloat16)
    x = torch.zeros(3, K, dtype=torch.bfloat16)
    for m, k in enumerate([0, 13, 39]):
        x[m, k] = 2.0
    y, _ = orc.gemm_bf16(_bits(x), _bits(w))
    for m, k in enumerate([0, 13, 39]):
        assert np.array_equal(y[m], 2.0 * w[:, k].double().numpy())
