"""The iteration-shaped batch: 96 rollouts x 4608 tokens = 442368 rows through a
FLUX.1-shaped linear chain 3072 -> 12288 -> 3072 (Sol-RL project page, "Two-Stage
Pipeline", Stage 1: N = 96 noises through the NVFP4-quantized solver; the chain's
shapes are those of the FLUX.1 MLP).

Parity, through the C ABI, against the oracle on sampled rows (rows are independent
in every step) plus the last row tile:
  * the down-projection (K = 12288) on its own, realistic operands, 4608 and 36864 rows;
  * the up-projection at the full 442368 rows, realistic operands;
  * the whole chain: act_quant(X) -> nvfp4_gemm -> bf16 hidden -> act_quant ->
    nvfp4_gemm, on the GPU for all rows.

The chain's inputs are built so that the first linear is exact on both sides, which
makes the bf16 hidden state bit-identical between the GPU and the oracle and lets the
second quantization be compared bit for bit:
  * every row of W_up is zero outside one 16-element block, so each output is a sum
    of 16 block-scaled E2M1 products, exact in fp32 (and in fp64);
  * one element of every row of X is +-336 = 2688 * 2^-3 (larger than any other
    element), so its per-row scale is exactly 2^-3; one element of W_up is
    2688 * 2^-12, so the per-tensor scale is exactly 2^-12; the products of the
    scales are then exact and y is rounded to bf16 once, identically on both sides.
The down-projection's weights are the realistic ones, merged with a rank-32 LoRA.
"""

import dataclasses

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import assert_gemm_close, np_, require_gpu, unswizzle_sf

pytestmark = pytest.mark.gpu


def _rows(M, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(M, n, replace=False), np.arange(M - 128, M)]))


def _oracle_weight(orc, cfg, W, A, B):
    Wn = workloads.bf16_bits(W) if W.dtype == torch.bfloat16 else W.numpy()
    return orc.requant(Wn, None if A is None else A.numpy(), None if B is None else B.numpy(),
                       workloads.LORA_ALPHA)


@pytest.mark.parametrize("M", [4608, 36864])
def test_iteration_down_projection(orc, M):
    """nvfp4_gemm at K = 12288, N = 3072 (the chain's second linear), realistic
    operands: one image (4608 rows) and 8 images (the full batch runs in the chain
    test below)."""
    require_gpu()
    cfg = dataclasses.replace(workloads.LINEARS["iter_down"], M=M)
    X = workloads.activations(cfg, seed=0)
    W = workloads.weight(cfg, seed=0)
    A, B = workloads.lora(cfg, seed=0)
    bias = workloads.bias(cfg, seed=0)
    w_q = nv.nvfp4_requant(W.cuda(), A.cuda(), B.cuda(), workloads.LORA_ALPHA)
    Xd = X.cuda()
    del X
    a_q = nv.nvfp4_act_quant(Xd)
    y = nv.nvfp4_gemm(a_q, w_q, bias.cuda())
    torch.cuda.synchronize()
    rows = _rows(M, 256, 11)
    y = np_(y[torch.from_numpy(rows).cuda()])
    xs = workloads.bf16_bits(Xd[torch.from_numpy(rows).cuda()].cpu())
    del Xd, a_q
    wc, wsf, ws = _oracle_weight(orc, cfg, W, A, B)
    ac, asf, a_s = orc.act_quant(xs)
    y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(bias))
    assert_gemm_close(y, y_ref, S, f"iter_down M={M}")
    assert nv.nvfp4_device_status() == 0


def test_iteration_up_projection_full_batch(orc):
    """nvfp4_gemm at the up-projection's full 442368 rows (3456 row tiles, the
    row-tile schedule at its largest), realistic operands, bias."""
    require_gpu()
    cfg = workloads.LINEARS["iter_up"]
    W = workloads.weight(cfg, seed=0)
    A, B = workloads.lora(cfg, seed=0)
    bias = workloads.bias(cfg, seed=0)
    X = workloads.activations(cfg, seed=0)
    w_q = nv.nvfp4_requant(W.cuda(), A.cuda(), B.cuda(), workloads.LORA_ALPHA)
    a_q = nv.nvfp4_act_quant(X.cuda())
    y = nv.nvfp4_gemm(a_q, w_q, bias.cuda())
    torch.cuda.synchronize()
    rows = _rows(cfg.M, 192, 12)
    y = np_(y[torch.from_numpy(rows).cuda()])
    wc, wsf, ws = _oracle_weight(orc, cfg, W, A, B)
    ac, asf, a_s = orc.act_quant(workloads.bf16_bits(X)[rows])
    y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws, workloads.bf16_bits(bias))
    assert_gemm_close(y, y_ref, S, "iter_up full batch")


def _chain_inputs(seed=0):
    up = workloads.LINEARS["iter_up"]
    M, K1, N1 = up.M, up.K, up.N
    # X: realistic activations, with one element per row set to +-336 (2688 * 2^-3);
    # the outlier channels reach ~30 * 6 = 180 at most, so 336 is each row's maximum.
    X = workloads.activations(up, seed=seed)
    g = torch.Generator().manual_seed(seed * 7919 + 1)
    pos = torch.randint(0, K1, (M,), generator=g)
    sign = torch.randint(0, 2, (M,), generator=g).to(torch.float32) * 2 - 1
    X[torch.arange(M), pos] = (336.0 * sign).to(torch.bfloat16)
    # W_up: realistic values kept in one 16-element block per row, zero elsewhere.
    W = workloads.weight(up, seed=seed).float()
    blk = torch.randint(0, K1 // 16, (N1,), generator=g)
    keep = torch.zeros(N1, K1 // 16, dtype=torch.bool)
    keep[torch.arange(N1), blk] = True
    W = torch.where(keep.repeat_interleave(16, dim=1), W, torch.zeros(())).clamp(-0.5, 0.5)
    W[0, int(blk[0]) * 16] = 2688.0 * 2.0 ** -12  # 0.65625: the tensor's maximum, exactly
    return X, W.to(torch.bfloat16)


def test_iteration_chain_sampled_rows(orc):
    """act_quant -> nvfp4_gemm (3072 -> 12288) -> bf16 hidden -> act_quant ->
    nvfp4_gemm (12288 -> 3072) for all 442368 rows on the GPU; on sampled rows the
    hidden state and its NVFP4 codes, scales and per-row scales are bit-identical to
    the oracle's, and the output is within the GEMM tolerance."""
    require_gpu()
    down = workloads.LINEARS["iter_down"]
    X, W_up = _chain_inputs()
    W_dn = workloads.weight(down, seed=0)
    A_dn, B_dn = workloads.lora(down, seed=0)
    bias_dn = workloads.bias(down, seed=0)
    M, K1, N1 = X.shape[0], X.shape[1], W_up.shape[0]
    rows = _rows(M, 128, 13)
    xs = workloads.bf16_bits(X[torch.from_numpy(rows)])

    # GPU: the whole chain for every row.
    w_up_q = nv.nvfp4_requant(W_up.cuda())          # no LoRA: the built weight itself
    w_dn_q = nv.nvfp4_requant(W_dn.cuda(), A_dn.cuda(), B_dn.cuda(), workloads.LORA_ALPHA)
    Xd = X.cuda()
    del X
    a_q = nv.nvfp4_act_quant(Xd)
    del Xd
    H = nv.nvfp4_gemm(a_q, w_up_q)                   # [M, 12288] bf16
    del a_q
    h_q = nv.nvfp4_act_quant(H)
    y = nv.nvfp4_gemm(h_q, w_dn_q, bias_dn.cuda())   # [M, 3072] bf16
    torch.cuda.synchronize()
    ridx = torch.from_numpy(rows).cuda()
    h_gpu = np_(H[ridx])
    hc_gpu = np_(h_q[0][ridx])
    hs_gpu = np_(h_q[2][ridx])
    hsf_rm, _ = unswizzle_sf(np_(h_q[1]), M, N1)
    hsf_gpu = hsf_rm[rows]
    y_gpu = np_(y[ridx])
    del H, h_q, y
    assert nv.nvfp4_device_status() == 0

    # Oracle: the same chain on the sampled rows.
    wc, wsf, ws = orc.requant(workloads.bf16_bits(W_up), None, None, workloads.LORA_ALPHA)
    assert ws[0] == np.float32(2.0 ** -12)
    ac, asf, a_s = orc.act_quant(xs)
    assert np.all(a_s == np.float32(2.0 ** -3))
    y1, _ = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, ws)
    # y1 is exact and fits fp32; bf16 round-to-nearest-even of it, once.
    h_ref = workloads.bf16_bits(torch.from_numpy(y1.astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(h_gpu, h_ref), f"hidden differs at {np.argwhere(h_gpu != h_ref)[:3]}"
    hc, hsf, hs = orc.act_quant(h_ref)
    assert np.array_equal(hs_gpu.view(np.uint32), hs.view(np.uint32)), "hidden per-row scales differ"
    assert np.array_equal(hsf_gpu, hsf), "hidden block scales differ"
    assert np.array_equal(hc_gpu, hc), "hidden codes differ"
    wdc, wdsf, wds = _oracle_weight(orc, down, W_dn, A_dn, B_dn)
    y_ref, S = orc.gemm_nvfp4(hc, hsf, hs, wdc, wdsf, wds, workloads.bf16_bits(bias_dn))
    assert_gemm_close(y_gpu, y_ref, S, "chain output")
