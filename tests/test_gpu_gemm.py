"""Parity of nvfp4_gemm and bf16_gemm (through the C ABI) with the oracle.

Tolerance (the task's stated bound): |y - y_oracle| <= 1e-3 * sum_k |a_k b_k|
+ 2^-8 |y_oracle|, the second term being the bf16 output rounding.  Checked on
all outputs for small and SANA-shaped problems and for random-operand problems
with ragged M/N/K tails, and on sampled rows plus the last row tile at the
FLUX.1- and SD3.5-L-shaped full sizes.  Operands fed to the oracle come from
the seeded generators or from the oracle's own quantizers, never from the GPU.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import assert_gemm_close, np_, require_gpu, swizzle_sf

pytestmark = pytest.mark.gpu


def _to_gpu_operand(codes, sf_rm, s, K):
    return (torch.from_numpy(codes).cuda(), torch.from_numpy(swizzle_sf(sf_rm, K)).cuda(),
            torch.from_numpy(np.ascontiguousarray(s, np.float32)).cuda())


@pytest.mark.parametrize("M,N,K,with_bias", [
    (128, 256, 256, True), (200, 264, 192, True), (1, 8, 64, False), (300, 520, 320, False),
    (129, 384, 1024, True), (2048, 2048, 2048, True),
])
def test_nvfp4_gemm_random_operands(orc, M, N, K, with_bias):
    require_gpu()
    ac, asf, a_s = [t.numpy() for t in workloads.random_nvfp4_operand(M, K, seed=M, stream=0)]
    wc, wsf, w_s = [t.numpy() for t in workloads.random_nvfp4_operand(N, K, seed=N, stream=1)]
    w_s = w_s[:1]
    bias = workloads.bias(workloads.LinearConfig("b", M=M, K=K, N=N), seed=K) if with_bias else None
    y = nv.nvfp4_gemm(_to_gpu_operand(ac, asf, a_s, K), _to_gpu_operand(wc, wsf, w_s, K),
                      None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, w_s,
                              None if bias is None else workloads.bf16_bits(bias))
    assert_gemm_close(np_(y), y_ref, S, f"nvfp4 {M}x{N}x{K}")


def test_nvfp4_gemm_extreme_scales(orc):
    """Largest and smallest scale bytes, all codes: no overflow in the fp32 path."""
    require_gpu()
    M, N, K = 256, 256, 512
    ac, asf, a_s = [t.numpy() for t in workloads.random_nvfp4_operand(M, K, 3, 0, sf_lo=0x00, sf_hi=0x7E)]
    wc, wsf, w_s = [t.numpy() for t in workloads.random_nvfp4_operand(N, K, 3, 1, sf_lo=0x00, sf_hi=0x7E)]
    y = nv.nvfp4_gemm(_to_gpu_operand(ac, asf, a_s, K), _to_gpu_operand(wc, wsf, w_s[:1], K))
    torch.cuda.synchronize()
    y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, w_s[:1])
    assert_gemm_close(np_(y), y_ref, S, "extreme scales")


def _pipeline(orc, name, rows=None, seed=0):
    """GPU: requant + act_quant + nvfp4_gemm; oracle: the same from the same seeds."""
    cfg = workloads.LINEARS[name]
    X = workloads.activations(cfg, seed=seed)
    W = workloads.weight(cfg, seed=seed)
    A, B = workloads.lora(cfg, seed=seed)
    bias = workloads.bias(cfg, seed=seed)
    w_q = nv.nvfp4_requant(W.cuda(), A.cuda(), B.cuda(), workloads.LORA_ALPHA)
    a_q = nv.nvfp4_act_quant(X.cuda())
    y = nv.nvfp4_gemm(a_q, w_q, bias.cuda())
    torch.cuda.synchronize()
    y = np_(y)
    Wn = workloads.bf16_bits(W) if W.dtype == torch.bfloat16 else W.numpy()
    wc, wsf, ws = orc.requant(Wn, A.numpy(), B.numpy(), workloads.LORA_ALPHA)
    xb = workloads.bf16_bits(X)
    if rows is None:
        ac, asf, a_s = orc.act_quant(xb)
        y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(bias))
        assert_gemm_close(y, y_ref, S, name)
    else:
        ac, asf, a_s = orc.act_quant(xb[rows])
        y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(bias))
        assert_gemm_close(y[rows], y_ref, S, name)


@pytest.mark.parametrize("name", ["tiny", "sana"])
def test_nvfp4_pipeline_all_outputs(orc, name):
    require_gpu()
    _pipeline(orc, name)


@pytest.mark.parametrize("name", ["flux_up", "sd35_qkv", "sd35_mlp"])
def test_nvfp4_pipeline_sampled_rows(orc, name):
    require_gpu()
    M = workloads.LINEARS[name].M
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(M, 192, replace=False), np.arange(M - 64, M)]))
    _pipeline(orc, name, rows=rows)


@pytest.mark.parametrize("M,N,K,with_bias", [
    (128, 256, 64, True), (200, 264, 200, True), (1, 8, 8, False), (333, 520, 136, True),
    (1024, 2304, 2240, True),
])
def test_bf16_gemm_shapes(orc, M, N, K, with_bias):
    require_gpu()
    g = torch.Generator().manual_seed(M + N + K)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    bias = (torch.randn(N, generator=g) * 0.02).to(torch.bfloat16) if with_bias else None
    y = nv.bf16_gemm(X.cuda(), W.cuda(), None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    y_ref, S = orc.gemm_bf16(workloads.bf16_bits(X), workloads.bf16_bits(W),
                             None if bias is None else workloads.bf16_bits(bias))
    assert_gemm_close(np_(y), y_ref, S, f"bf16 {M}x{N}x{K}")


def test_bf16_gemm_flux_sampled_rows(orc):
    require_gpu()
    cfg = workloads.LINEARS["flux_up"]
    X = workloads.activations(cfg)
    W = workloads.weight(cfg)
    bias = workloads.bias(cfg)
    y = np_(nv.bf16_gemm(X.cuda(), W.cuda(), bias.cuda()))
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([rng.choice(cfg.M, 64, replace=False), np.arange(cfg.M - 16, cfg.M)]))
    y_ref, S = orc.gemm_bf16(workloads.bf16_bits(X), workloads.bf16_bits(W), workloads.bf16_bits(bias),
                             rows=rows)
    assert_gemm_close(y[rows], y_ref, S, "bf16 flux")


def test_gemm_does_not_write_outside_y():
    require_gpu()
    M, N, K = 130, 264, 128
    ac, asf, a_s = [t.numpy() for t in workloads.random_nvfp4_operand(M, K, 1, 0)]
    wc, wsf, w_s = [t.numpy() for t in workloads.random_nvfp4_operand(N, K, 1, 1)]
    buf = torch.full((M * N + 4096,), 12345, dtype=torch.int16, device="cuda")
    out = buf[: M * N].view(torch.bfloat16).view(M, N)
    nv.nvfp4_gemm(_to_gpu_operand(ac, asf, a_s, K), _to_gpu_operand(wc, wsf, w_s[:1], K), out=out)
    torch.cuda.synchronize()
    assert bool((buf[M * N:] == 12345).all())
