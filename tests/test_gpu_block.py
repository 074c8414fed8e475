"""The synthetic DiT block (reading R15 of oracle/oracle.c's header; Sol-RL project
page, "Two-Stage Pipeline", Stage 1: the NVFP4-quantized solver runs the DiT's linears
in NVFP4): its streaming steps, its attention and the whole block against the oracle.

The softmax and the GELU run in fp32 on the GPU and in double in the oracle, and the
attention's logits and products accumulate in fp32 on the tensor cores against exact
sums in the oracle: rounded to bf16, results agree except where a value falls within
the fp32 error of a bf16 midpoint, where they differ by one bf16 step.  The tests bound
both the size and the share of those differences.  The residual add is exact.  The
block is then compared as a whole: a one-step difference in an activation can move an
NVFP4 code or a row scale downstream, so it is held to a tolerance on the output
(stated in each test; at the FLUX.1 shape one derived from the activation
quantization's own effect), and its residual wiring bit for bit.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import oracle as orc
import workloads
from gpu_util import np_, require_gpu

pytestmark = pytest.mark.gpu


def _bf16(a, dev="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(orc.bf16_rne(a)).view(np.int16)).view(torch.bfloat16)
    return t.to(dev)


def _ulp_steps(got_bits, ref_bits):
    """Distance in bf16 steps between two arrays of bf16 patterns (same signs assumed
    where they differ by a step; a sign change counts as large)."""
    g = got_bits.astype(np.int32)
    r = ref_bits.astype(np.int32)
    same_sign = (g & 0x8000) == (r & 0x8000)
    d = np.abs((g & 0x7FFF) - (r & 0x7FFF))
    zero_pair = ((g & 0x7FFF) == 0) & ((r & 0x7FFF) == 0)
    return np.where(same_sign | zero_pair, d, 1 << 16)


@pytest.mark.parametrize("rows,cols", [(64, 256), (300, 4608)])
def test_softmax_rows(rows, cols):
    require_gpu()
    rng = np.random.default_rng(rows + cols)
    L = rng.standard_normal((rows, cols)) * 6
    scale = float(np.float32(1 / np.sqrt(128)))
    Ld = _bf16(L)
    P = np_(nv.bf16_softmax_rows(Ld, scale))
    ref = orc.softmax_bf16(np_(Ld), scale)
    steps = _ulp_steps(P, ref)
    assert steps.max() <= 1, steps.max()
    assert (steps > 0).mean() < 2e-3, (steps > 0).mean()
    # In place gives the same bits.
    nv.bf16_softmax_rows(Ld, scale, P=Ld)
    assert np.array_equal(np_(Ld), P)


def test_gelu_and_add():
    require_gpu()
    rng = np.random.default_rng(7)
    x = rng.standard_normal(1 << 20) * 10.0 ** rng.uniform(-3, 1.2, 1 << 20)
    xd = _bf16(x)
    g = np_(nv.bf16_gelu(xd))
    ref = orc.gelu_bf16(np_(xd))
    steps = _ulp_steps(g, ref)
    assert steps.max() <= 1 and (steps > 0).mean() < 2e-3, (steps.max(), (steps > 0).mean())
    yd = _bf16(rng.standard_normal(1 << 20) * 10.0 ** rng.uniform(-4, 4, 1 << 20))
    s = np_(nv.bf16_add(xd, yd))
    assert np.array_equal(s, orc.add_bf16(np_(xd), np_(yd)))


@pytest.mark.parametrize("B,S,D,H", [(2, 256, 256, 2), (1, 512, 384, 3), (2, 320, 256, 4), (3, 192, 128, 1), (2, 64, 128, 2),
                                     (1, 4608, 256, 2)])
def test_attention(B, S, D, H):
    """The fused attention kernel: head widths 128 and 64, several 256-row query blocks,
    S % 256 != 0 (a query block with rows past S in one or both CTAs, and a last key
    tile of 64, 128 or 192 valid keys, some column slices wholly masked), and 4608 keys
    (18 tiles, both passes around the rings)."""
    require_gpu()
    rng = np.random.default_rng(B * S + D)
    qkv = _bf16(rng.standard_normal((B * S, 3 * D)) * 0.5)
    o = np_(nv.nvfp4_dit_attention(qkv, B, S, H))
    ref = orc.attention(np_(qkv), B, S, H)
    steps = _ulp_steps(o, ref)
    assert (steps == 0).mean() > 0.95, (steps == 0).mean()
    vo, vr = orc.bf16_value(o), orc.bf16_value(ref)
    assert np.max(np.abs(vo - vr)) <= 2.0 ** -6 * np.max(np.abs(vr))
    assert nv.nvfp4_device_status() == 0


def _weights(rng, D, scale=0.03, zero=()):
    shapes = {"qkv": (3 * D, D), "o": (D, D), "up": (4 * D, D), "dn": (D, 4 * D)}
    w_bits, b_bits = {}, {}
    for k, (n, kk) in shapes.items():
        w_bits[k] = np.zeros((n, kk), np.uint16) if k in zero else orc.bf16_rne(rng.standard_normal((n, kk)) * scale)
        b_bits[k] = None if k in zero else orc.bf16_rne(rng.standard_normal(n) * 0.02)
    return w_bits, b_bits


def _gpu_weights(w_bits, b_bits):
    out = []
    for k in ("qkv", "o", "up", "dn"):
        W = torch.from_numpy(w_bits[k].view(np.int16)).view(torch.bfloat16).cuda()
        codes, sf, s_t = nv.nvfp4_requant(W)
        bias = None if b_bits[k] is None else torch.from_numpy(b_bits[k].view(np.int16)).view(torch.bfloat16).cuda()
        out.append((codes, sf, s_t, bias))
    return out


def _oracle_weights(w_bits):
    return {k: orc.requant(w_bits[k], None, None, 32.0) for k in w_bits}


def _block_tolerance(vo, vr):
    rms = np.sqrt(np.mean(vr ** 2))
    assert np.linalg.norm(vo - vr) <= 2.0 ** -7 * np.linalg.norm(vr)
    assert (np.abs(vo - vr) <= 2.0 ** -5 * np.abs(vr) + 2.0 ** -8 * rms).mean() >= 0.99


@pytest.mark.parametrize("B,S,D,H", [(1, 256, 512, 4), (2, 128, 256, 2), (3, 64, 256, 4)])
def test_block_against_oracle(B, S, D, H):
    """Tolerance: relative Frobenius error of the output below 2^-7, and 99% of
    elements within 2^-5 |ref| + 2^-8 rms(ref).  B = 3, S = 64: 192 tokens, a partial
    GEMM tile and dh = 64."""
    require_gpu()
    rng = np.random.default_rng(11 * B + S)
    x = orc.bf16_rne(rng.standard_normal((B * S, D)))
    w_bits, b_bits = _weights(rng, D)
    out = np_(nv.nvfp4_dit_block(_bf16(orc.bf16_value(x)), B, S, H, _gpu_weights(w_bits, b_bits)))
    ref = orc.dit_block(x, _oracle_weights(w_bits), b_bits, B, S, H)["out"]
    _block_tolerance(orc.bf16_value(out), orc.bf16_value(ref))
    assert nv.nvfp4_device_status() == 0


def test_block_flux_shape_sampled_rows():
    """The FLUX.1-shaped block as the benchmark runs it (8 images x 4608 tokens, D 3072,
    24 heads, the seeded block workload): 32 rows of the last image, its first and last
    token included, against the oracle's row-restricted block.

    Tolerance.  Each stage of the GPU block agrees with the oracle's stage to the
    rounding of its fp32 accumulations (attention logits, softmax, products), but the
    next linear's activation quantizer turns a few of those one-step differences into a
    different E2M1 code (or block or row scale), and one changed code moves a whole
    output row by about a percent; three linears deep that reaches some percent.  So a
    sampled row either matches bit for bit or differs by about what the activation
    quantization itself does to it.  The test asks (a) at least 40% of the rows bit for
    bit equal, (b) every row within 2x the distance between the oracle's row and the
    same block with unquantized activations (two sets of code decisions on nearly equal
    inputs each stay about that far from the unquantized result), (c) the relative
    Frobenius error over the rows below 2^-4."""
    require_gpu()
    cfg = workloads.BLOCKS["flux"]
    x = workloads.block_input(cfg, seed=0)
    wts = workloads.block_weights(cfg, seed=0)
    gpu_w = []
    for name in workloads.BLOCK_LINEARS:
        W, b = wts[name]
        codes, sf, s_t = nv.nvfp4_requant(W.cuda())
        gpu_w.append((codes, sf, s_t, b.cuda()))
    out = nv.nvfp4_dit_block(x.cuda(), cfg.B, cfg.S, cfg.H, gpu_w)
    last = (cfg.B - 1) * cfg.S
    rows = np.concatenate([[last, last + cfg.S - 1],
                           last + np.random.default_rng(7).choice(np.arange(1, cfg.S - 1), 30, replace=False)])
    got = workloads.bf16_bits(out[torch.from_numpy(rows).cuda()].cpu())
    assert nv.nvfp4_device_status() == 0
    del out, gpu_w
    w_o = {k: orc.requant(workloads.bf16_bits(wts[k][0]), None, None, 32.0) for k in workloads.BLOCK_LINEARS}
    b_o = {k: workloads.bf16_bits(wts[k][1]) for k in workloads.BLOCK_LINEARS}
    xb = workloads.bf16_bits(x)
    ref = orc.dit_block_rows(xb, w_o, b_o, cfg.B, cfg.S, cfg.H, rows)
    unq = orc.dit_block_rows(xb, w_o, b_o, cfg.B, cfg.S, cfg.H, rows, quantize_activations=False)
    vg, vr, vu = orc.bf16_value(got), orc.bf16_value(ref), orc.bf16_value(unq)
    d_gpu = np.linalg.norm(vg - vr, axis=1)
    d_quant = np.linalg.norm(vr - vu, axis=1)
    exact = np.all(got == ref, axis=1)
    info = (exact.mean(), np.round(d_gpu / np.linalg.norm(vr, axis=1), 4),
            np.round(d_quant / np.linalg.norm(vr, axis=1), 4))
    assert exact.mean() >= 0.4, info
    assert np.all(d_gpu <= 2.0 * d_quant), info
    assert np.linalg.norm(vg - vr) <= 2.0 ** -4 * np.linalg.norm(vr), info


@pytest.mark.parametrize("B,S,D,H", [(2, 128, 256, 2), (1, 320, 512, 4), (3, 64, 256, 4)])
def test_block_equals_its_public_steps(B, S, D, H):
    """The block fuses the GELU and both residual adds into the GEMM epilogues; the result
    must equal, bit for bit, the same block composed from the library's public calls
    (act_quant, nvfp4_gemm, the attention, bf16_gelu, bf16_add)."""
    require_gpu()
    rng = np.random.default_rng(3 * B + S)
    x = _bf16(rng.standard_normal((B * S, D)))
    w_bits, b_bits = _weights(rng, D)
    w = _gpu_weights(w_bits, b_bits)

    def lin(a, wi):
        return nv.nvfp4_gemm(nv.nvfp4_act_quant(a), wi[:3], bias=wi[3])
    qkv = lin(x, w[0])
    h1 = nv.bf16_add(lin(nv.nvfp4_dit_attention(qkv, B, S, H), w[1]), x)
    ref = nv.bf16_add(lin(nv.bf16_gelu(lin(h1, w[2])), w[3]), h1)
    out = nv.nvfp4_dit_block(x, B, S, H, w)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert nv.nvfp4_device_status() == 0


def test_block_residual_wiring_is_exact():
    """Zero output projections: the GPU block returns its input bit for bit."""
    require_gpu()
    rng = np.random.default_rng(5)
    B, S, D, H = 2, 128, 256, 2
    x = _bf16(rng.standard_normal((B * S, D)))
    w_bits, b_bits = _weights(rng, D, zero=("o", "dn"))
    out = nv.nvfp4_dit_block(x, B, S, H, _gpu_weights(w_bits, b_bits))
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))


def test_block_shape_rules():
    require_gpu()
    assert nv.dit_block_workspace_bytes(1, 100, 256, 2) == 0      # S % 64
    assert nv.dit_block_workspace_bytes(1, 128, 256, 3) == 0      # H does not divide D into 64s
    assert nv.dit_block_workspace_bytes(1, 128, 384, 2) == 0      # dh = 192: the attention takes 64 or 128
    assert nv.dit_attention_workspace_bytes(2, 320, 256, 4) == 2 * 320 * 256 * 2  # v transposed
    assert nv.dit_block_workspace_bytes(8, 4608, 3072, 24) > 0
