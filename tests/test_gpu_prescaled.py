"""Per-token activation quantization with the row scales handed over by the producing
GEMM (Sol-RL project page, "Two-Stage Pipeline", Stage 1: the NVFP4-quantized solver
quantizes every linear's input per token).

nvfp4_gemm_rowamax writes max_n |Y[m, n]| of its bf16 output; nvfp4_act_quant_prescaled
then quantizes Y in one streaming pass.  The results must be bit-identical to
nvfp4_act_quant on the same Y (which is pinned to the oracle elsewhere), and to the
oracle on sampled rows directly.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import np_, require_gpu, unswizzle_sf

pytestmark = pytest.mark.gpu


def _operands(M, N, K, seed):
    cfg = workloads.LinearConfig(name="prescaled", M=M, K=K, N=N, w_outlier_frac=0.01, w_outlier_gain=8.0,
                                 x_outlier_frac=0.01, x_outlier_gain=30.0)
    X = workloads.activations(cfg, seed=seed).cuda()
    W = workloads.weight(cfg, seed=seed).cuda()
    bias = workloads.bias(cfg, seed=seed).cuda()
    return nv.nvfp4_act_quant(X), nv.nvfp4_requant(W), bias


def _same(a, b, what):
    a, b = np_(a), np_(b)
    assert np.array_equal(a, b), f"{what} differ at {np.argwhere(a != b)[:3]}"


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 520, 3072), (4608, 12288, 3072), (130, 3072, 12288)])
def test_gemm_rowamax(M, N, K):
    """Y is nvfp4_gemm's, bit for bit; row_amax is max |Y| per row, exactly."""
    require_gpu()
    a_q, w_q, bias = _operands(M, N, K, seed=M + N)
    y_ref = nv.nvfp4_gemm(a_q, w_q, bias)
    y, amax = nv.nvfp4_gemm_rowamax(a_q, w_q, bias)
    torch.cuda.synchronize()
    _same(y, y_ref, "Y")
    exp = y.float().abs().amax(dim=1)
    _same(amax, exp, "row amax")
    # A second call into the same buffer starts from zero again.
    y2, amax2 = nv.nvfp4_gemm_rowamax(a_q, w_q, None, out=y, row_amax=amax)
    torch.cuda.synchronize()
    _same(amax2, nv.nvfp4_gemm(a_q, w_q).float().abs().amax(dim=1), "row amax, second call")
    assert nv.nvfp4_device_status() == 0


def test_gemm_rowamax_empty_output_columns():
    require_gpu()
    a_q, w_q, _ = _operands(64, 256, 256, seed=1)
    empty_w = (w_q[0][:0], w_q[1], w_q[2])
    amax = torch.full((64,), 7.0, device="cuda")
    y, amax = nv.nvfp4_gemm_rowamax(a_q, empty_w, row_amax=amax)
    torch.cuda.synchronize()
    assert y.shape == (64, 0) and not amax.any()


def _check_prescaled(orc, X, rows):
    M, K = X.shape
    amax = X.float().abs().amax(dim=1)
    c, sf, s = nv.nvfp4_act_quant_prescaled(X, amax)
    c_ref, sf_ref, s_ref = nv.nvfp4_act_quant(X)
    torch.cuda.synchronize()
    _same(c, c_ref, "codes")
    _same(sf, sf_ref, "scales (padding rows included)")
    _same(s, s_ref, "s_row")
    # And the oracle on sampled rows.
    sf_rm, sf_pad = unswizzle_sf(np_(sf), M, K)
    assert not sf_pad.any()
    oc, osf, os_ = orc.act_quant(workloads.bf16_bits(X[torch.from_numpy(rows).cuda()].cpu()))
    assert np.array_equal(np_(c)[rows], oc)
    assert np.array_equal(sf_rm[rows], osf)
    assert np.array_equal(np_(s)[rows].view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("name,M", [("flux_up", 36864), ("iter_down", 4608), ("sana", 1000), ("flux_up", 1),
                                    ("sd35_qkv", 130)])
def test_act_quant_prescaled(orc, name, M):
    require_gpu()
    cfg = workloads.LINEARS[name]
    X = workloads.activations(cfg, seed=5, rows=M).cuda()
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([rng.choice(M, min(M, 96), replace=False), [M - 1]]))
    _check_prescaled(orc, X, rows)


def test_act_quant_prescaled_edge_values(orc):
    """Zero rows, a row of one nonzero, subnormal-scale rows, ties of E2M1 midpoints."""
    require_gpu()
    M, K = 64, 2240
    g = torch.Generator().manual_seed(3)
    X = torch.randn(M, K, generator=g) * 0.02
    X[0] = 0.0
    X[1] = 0.0
    X[1, 17] = -3.0
    X[2] *= 1e-30
    X[3] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * (K // 8)) * (1 - 2 * (torch.arange(K) % 3 == 0))
    X = X.to(torch.bfloat16).cuda()
    _check_prescaled(orc, X, np.arange(M))


def test_chain_with_handed_over_row_scales(orc):
    """act_quant -> nvfp4_gemm_rowamax -> act_quant_prescaled on the FLUX.1 MLP
    up-projection (4608 tokens): the hidden state's NVFP4 form is the one
    nvfp4_act_quant gives, on every row, and the oracle's on sampled rows."""
    require_gpu()
    cfg = workloads.LINEARS["flux_up"]
    X = workloads.activations(cfg, seed=2, rows=4608).cuda()
    W = workloads.weight(cfg, seed=2).cuda()
    A, B = [t.cuda() for t in workloads.lora(cfg, seed=2)]
    w_q = nv.nvfp4_requant(W, A, B, workloads.LORA_ALPHA)
    H, amax = nv.nvfp4_gemm_rowamax(nv.nvfp4_act_quant(X), w_q, workloads.bias(cfg, seed=2).cuda())
    rows = np.unique(np.concatenate([np.random.default_rng(9).choice(4608, 64, replace=False), [4607]]))
    _check_prescaled(orc, H, rows)
    c, sf, s = nv.nvfp4_act_quant_prescaled(H, amax)
    c_ref, sf_ref, s_ref = nv.nvfp4_act_quant(H)
    torch.cuda.synchronize()
    _same(c, c_ref, "hidden codes")
    _same(sf, sf_ref, "hidden scales")
    _same(s, s_ref, "hidden s_row")
    assert nv.nvfp4_device_status() == 0
