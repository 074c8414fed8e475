"""Parity of nvfp4_act_quant and nvfp4_requant (through the C ABI) with the oracle.

Codes, scales and second-level scales must match bit for bit, on seeded
synthetic inputs of every configuration (FLUX.1-, SD3.5-L- and SANA-shaped
linears at full size; the iteration-shaped batch on sampled rows) and on the
edge cases: one row, ragged row counts, all-zero and constant rows, huge and
tiny magnitudes (subnormal and zero block scales), exact grid values, negative
zeros, ranks 0 / 1 / 7 / 64.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import np_, require_gpu, unswizzle_sf

pytestmark = pytest.mark.gpu


def _check_act(orc, X_cpu, rows=None):
    """Runs act_quant on the GPU for all of X and compares `rows` (default all)."""
    M, K = X_cpu.shape
    codes, sf, s = nv.nvfp4_act_quant(X_cpu.cuda())
    torch.cuda.synchronize()
    codes, sf, s = np_(codes), np_(sf), np_(s)
    sf_rm, sf_pad = unswizzle_sf(sf, M, K)
    assert not sf_pad.any(), "scale padding rows must be zero"
    bits = workloads.bf16_bits(X_cpu)
    if rows is not None:
        bits = bits[rows]
        codes, sf_rm, s = codes[rows], sf_rm[rows], s[rows]
    oc, osf, os_ = orc.act_quant(bits)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)), "per-row scales differ"
    assert np.array_equal(sf_rm, osf), f"block scales differ at {np.argwhere(sf_rm != osf)[:3]}"
    assert np.array_equal(codes, oc), f"codes differ at {np.argwhere(codes != oc)[:3]}"


@pytest.mark.parametrize("name", ["tiny", "sana", "flux_up", "sd35_qkv"])
def test_act_quant_configs(orc, name):
    require_gpu()
    cfg = workloads.LINEARS[name]
    _check_act(orc, workloads.activations(cfg, seed=0))


def test_act_quant_iteration_batch_sampled_rows(orc):
    """442368 x 3072 (the iteration-shaped batch) on the GPU; 2048 sampled rows
    plus the last 128 checked (rows are independent)."""
    require_gpu()
    cfg = workloads.LINEARS["iter_up"]
    X = workloads.activations(cfg, seed=0)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(cfg.M, 2048, replace=False),
                                     np.arange(cfg.M - 128, cfg.M)]))
    _check_act(orc, X, rows)


@pytest.mark.parametrize("M,K", [(1, 64), (129, 128), (300, 12288), (77, 32768), (1000, 2240),
                                 (64, 512), (33, 4096), (130, 1536)])
def test_act_quant_shapes(orc, M, K):
    require_gpu()
    g = torch.Generator().manual_seed(M * 7 + K)
    X = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g) * 3)).to(torch.bfloat16)
    _check_act(orc, X)


def test_act_quant_edge_values(orc):
    require_gpu()
    K = 256
    g = torch.Generator().manual_seed(5)
    X = torch.randn(12, K, generator=g)
    X[0] = 0.0                                   # zero row: s = 0, all scales and codes 0
    X[1] = 0.37                                  # constant row
    X[2] *= 1e-36                                # tiny: subnormal block scales
    X[3, :16] = 1e4; X[3, 16:] = 1e-3            # blocks whose scale rounds to 0
    X[4] = -0.0                                  # negative zeros
    X[5] *= 3e38 / 4                             # near the top of the bf16 range
    X[6, ::2] = 0.0
    grid = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 6])
    X[7] = grid.repeat(K // 16) * 2.0 ** -5      # exact grid values (exact-division path)
    X[8] = torch.linspace(-6, 6, K)
    X[9, 0] = 1e30; X[9, 1:] = 1.0                # one huge outlier
    X[10] = torch.randn(K, generator=g) * 1e-20
    X[11, :] = 2.0 ** -133                        # bf16 subnormal-range inputs
    _check_act(orc, X.to(torch.bfloat16))


def test_act_quant_zero_rows_is_noop():
    require_gpu()
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    codes = torch.empty(0, 32, dtype=torch.uint8, device="cuda")
    sf = torch.empty(0, dtype=torch.uint8, device="cuda")
    s = torch.empty(0, dtype=torch.float32, device="cuda")
    nv.nvfp4_act_quant(X, codes, sf, s)


def _check_requant(orc, W, A, B, alpha, rows=None):
    N, K = W.shape
    codes, sf, s_t = nv.nvfp4_requant(W.cuda(), None if A is None else A.cuda(),
                                      None if B is None else B.cuda(), alpha)
    torch.cuda.synchronize()
    codes, sf, s_t = np_(codes), np_(sf), np_(s_t)
    sf_rm, sf_pad = unswizzle_sf(sf, N, K)
    assert not sf_pad.any(), "scale padding rows must be zero"
    Wn = workloads.bf16_bits(W) if W.dtype == torch.bfloat16 else W.numpy()
    oc, osf, os_ = orc.requant(Wn, None if A is None else A.numpy(), None if B is None else B.numpy(), alpha)
    assert s_t.view(np.uint32)[0] == os_.view(np.uint32)[0], f"s_t {s_t[0]!r} vs {os_[0]!r}"
    assert np.array_equal(sf_rm, osf), f"block scales differ at {np.argwhere(sf_rm != osf)[:3]}"
    assert np.array_equal(codes, oc), f"codes differ at {np.argwhere(codes != oc)[:3]}"


@pytest.mark.parametrize("name", ["tiny", "sana", "flux_up", "sd35_qkv", "sd35_mlp"])
def test_requant_configs(orc, name):
    require_gpu()
    cfg = workloads.LINEARS[name]
    W = workloads.weight(cfg, seed=0)
    A, B = workloads.lora(cfg, seed=0)
    _check_requant(orc, W, A, B, workloads.LORA_ALPHA)


def test_requant_iteration_down_projection(orc):
    """The down-projection shape of the iteration-shaped chain: [3072, 12288]."""
    require_gpu()
    cfg = workloads.LINEARS["iter_down"]
    W = workloads.weight(cfg, seed=1)
    A, B = workloads.lora(cfg, seed=1)
    _check_requant(orc, W, A, B, workloads.LORA_ALPHA)


def test_act_quant_per_tensor_variant(orc):
    """One per-tensor scale for activations: nvfp4_requant with no LoRA factors on
    FLUX-shaped bf16 activations (outlier channels included), 2048 rows."""
    require_gpu()
    X = workloads.activations(workloads.LINEARS["flux_up"], rows=2048)
    _check_requant(orc, X, None, None, workloads.LORA_ALPHA)


def _check_act_tensor(orc, X):
    M, K = X.shape
    codes, sf, s_t = nv.nvfp4_act_quant_tensor(X.cuda())
    torch.cuda.synchronize()
    codes, sf, s_t = np_(codes), np_(sf), np_(s_t)
    sf_rm, sf_pad = unswizzle_sf(sf, M, K)
    assert not sf_pad.any(), "scale padding rows must be zero"
    oc, osf, os_ = orc.requant(workloads.bf16_bits(X), None, None, workloads.LORA_ALPHA)
    assert s_t.view(np.uint32)[0] == os_.view(np.uint32)[0], f"s_t {s_t[0]!r} vs {os_[0]!r}"
    assert np.array_equal(sf_rm, osf), f"block scales differ at {np.argwhere(sf_rm != osf)[:3]}"
    assert np.array_equal(codes, oc), f"codes differ at {np.argwhere(codes != oc)[:3]}"


@pytest.mark.parametrize("M,K", [(2048, 3072), (1, 64), (300, 12288), (77, 32768), (129, 2240)])
def test_act_quant_tensor(orc, M, K):
    """nvfp4_act_quant_tensor (per-tensor scale, two passes) against the oracle's
    per-tensor quantization; FLUX-shaped activations for the first case."""
    require_gpu()
    if (M, K) == (2048, 3072):
        X = workloads.activations(workloads.LINEARS["flux_up"], rows=M)
    else:
        g = torch.Generator().manual_seed(M * 13 + K)
        X = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g) * 3)).to(torch.bfloat16)
    _check_act_tensor(orc, X)


def test_act_quant_tensor_edge_values(orc):
    require_gpu()
    g = torch.Generator().manual_seed(9)
    _check_act_tensor(orc, torch.zeros(130, 128, dtype=torch.bfloat16))   # zero tensor: s_t = 0
    X = torch.randn(64, 256, generator=g)
    X[5, 17] = -3e38                                                      # amax from a negative value
    X[7] = 2.0 ** -133
    _check_act_tensor(orc, X.to(torch.bfloat16))


@pytest.mark.parametrize("r", [0, 1, 7, 64])
def test_requant_ranks(orc, r):
    require_gpu()
    g = torch.Generator().manual_seed(r)
    N, K = 200, 320
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    if r == 0:
        _check_requant(orc, W, None, None, 32.0)
        return
    A = torch.randn(r, K, generator=g) / 32
    B = torch.randn(N, r, generator=g) * 0.01
    _check_requant(orc, W, A, B, 3.0)  # alpha / r not a power of two


def test_requant_edge_values(orc):
    require_gpu()
    g = torch.Generator().manual_seed(9)
    N, K = 131, 192
    W = torch.randn(N, K, generator=g) * 0.02
    W[0] = 0.0
    W[1] = -0.0
    W[2, :16] = 5.0
    W[3] *= 1e-30
    W[4, 0] = -1e3
    A = torch.randn(32, K, generator=g) / 32
    B = torch.randn(N, 32, generator=g) * 0.01
    B[0] = 0.0
    B[1] = 0.0   # row 1 stays -0 + 0 * ...
    _check_requant(orc, W.contiguous(), A, B, 32.0)
    _check_requant(orc, W.to(torch.bfloat16), A, B, 32.0)
    _check_requant(orc, torch.zeros(N, K), A * 0, B * 0, 32.0)


@pytest.mark.parametrize("N,K", [(1, 64), (100, 64), (257, 192), (640, 1088), (1024, 12288)])
def test_requant_tensor_core_shapes(orc, N, K):
    """bf16 weights with a rank-32 update take the tensor-core merge: one row, a
    256-row block whose second half is empty, ragged rows with a half-width last
    strip, and several row blocks per CTA pair (rows of B kept across strips)."""
    require_gpu()
    g = torch.Generator().manual_seed(N * 7 + K)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    A = torch.randn(32, K, generator=g) / 32
    B = torch.randn(N, 32, generator=g) * 0.01
    _check_requant(orc, W, A, B, 32.0)


def test_requant_tensor_core_degenerate(orc):
    """The tensor-core merge's degenerate cases: alpha = 0 (W' = W up to the sign of
    zero, which the chain's accumulator decides), zero rows of B and zero columns of
    A, an update far larger than W (most decisions fall to the exact chain), and
    factors whose products are fp32 subnormals."""
    require_gpu()
    g = torch.Generator().manual_seed(31)
    N, K = 300, 256
    W = torch.randn(N, K, generator=g) * 0.02
    W[0] = -0.0
    W[1, ::2] = -0.0
    W[1, 1::2] = 0.0
    W = W.to(torch.bfloat16)
    A = torch.randn(32, K, generator=g) / 32
    B = torch.randn(N, 32, generator=g) * 0.01
    B[2] = 0.0
    A[:, 5] = 0.0
    _check_requant(orc, W, A, B, 0.0)
    _check_requant(orc, W, A, B, 32.0)
    Wt = (torch.randn(N, K, generator=g) * 1e-6).to(torch.bfloat16)
    _check_requant(orc, Wt, torch.randn(32, K, generator=g), torch.randn(N, 32, generator=g), 32.0)
    Ws = (torch.randn(N, K, generator=g) * 1e-39).to(torch.bfloat16)
    _check_requant(orc, Ws, torch.randn(32, K, generator=g) * 1e-20,
                   torch.randn(N, 32, generator=g) * 1e-19, 32.0)


def test_requant_repeated_calls_reset_amax(orc):
    """s_t doubles as the amax accumulator: a second call on a smaller tensor must
    not see the first call's amax."""
    require_gpu()
    g = torch.Generator().manual_seed(11)
    W1 = torch.randn(64, 128, generator=g) * 10
    W2 = torch.randn(64, 128, generator=g) * 0.1
    codes = torch.empty(64, 64, dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.sf_bytes(64, 128), dtype=torch.uint8, device="cuda")
    s_t = torch.empty(1, device="cuda")
    nv.nvfp4_requant(W1.cuda(), codes=codes, sf=sf, s_t=s_t)
    nv.nvfp4_requant(W2.cuda(), codes=codes, sf=sf, s_t=s_t)
    _, _, os_ = orc.requant(W2.numpy(), None, None, 32.0)
    assert np_(s_t)[0] == os_[0]


def _check_merge(orc, W, A, B, alpha):
    """The GPU's merged weights (the values requant quantizes) against the
    oracle's fma chain, bit for bit."""
    got = np_(nv.nvfp4_test_merge(W.cuda(), None if A is None else A.cuda(),
                                  None if B is None else B.cuda(), alpha))
    Wn = workloads.bf16_bits(W) if W.dtype == torch.bfloat16 else W.numpy()
    want = orc.merge(Wn, None if A is None else A.numpy(), None if B is None else B.numpy(), alpha)
    bad = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, f"{len(bad)} merged values differ, first at {bad[:3]}"


@pytest.mark.parametrize("name", ["tiny", "sana", "flux_up"])
def test_merge_configs_bit_exact(orc, name):
    require_gpu()
    cfg = workloads.LINEARS[name]
    W = workloads.weight(cfg, seed=0)
    A, B = workloads.lora(cfg, seed=0)
    _check_merge(orc, W, A, B, workloads.LORA_ALPHA)


@pytest.mark.parametrize("r", [0, 1, 7, 33, 64])
@pytest.mark.parametrize("wdt", [torch.bfloat16, torch.float32])
def test_merge_ranks_and_tails(orc, r, wdt):
    """Ragged rows (200 = 3 row tiles + 8) and a half-width last strip (K = 320)."""
    require_gpu()
    g = torch.Generator().manual_seed(100 + r)
    N, K = 200, 320
    W = (torch.randn(N, K, generator=g) * 0.02).to(wdt)
    A = torch.randn(r, K, generator=g) / 32 if r else None
    B = torch.randn(N, r, generator=g) * 0.01 if r else None
    _check_merge(orc, W, A, B, 3.0)


def test_requant_amax_moved_by_lora(orc):
    """The largest |W'| is not at the largest |W|: a rank-1 update lifts another
    element of the same warp's rows above it, and, in a second case, one in a
    different CTA's tile."""
    require_gpu()
    N, K = 256, 512
    g = torch.Generator().manual_seed(21)
    W = torch.randn(N, K, generator=g) * 0.01
    W[5, 7] = 0.1
    W[9, 3] = -0.099
    A = torch.zeros(1, K)
    B = torch.zeros(N, 1)
    A[0, 3] = -0.005
    B[9, 0] = 1.0
    _check_requant(orc, W, A, B, 1.0)
    W2 = W.clone()
    W2[9, 3] = 0.0
    W2[200, 400] = 0.0995
    A2 = torch.zeros(1, K)
    B2 = torch.zeros(N, 1)
    A2[0, 400] = 0.001
    B2[200, 0] = 1.0
    _check_requant(orc, W2, A2, B2, 1.0)


def test_requant_lora_dominated(orc):
    """|B A| much larger than |W| everywhere (every element is a candidate for the
    maximum), and W constant in magnitude with mixed signs."""
    require_gpu()
    g = torch.Generator().manual_seed(22)
    N, K = 192, 256
    W = torch.randn(N, K, generator=g) * 1e-6
    A = torch.randn(32, K, generator=g)
    B = torch.randn(N, 32, generator=g)
    _check_requant(orc, W, A, B, 32.0)
    Wc = torch.full((N, K), 0.05) * torch.sign(torch.randn(N, K, generator=g))
    _check_requant(orc, Wc.to(torch.bfloat16), A / 32 * 0.01, B * 0.01, 32.0)


def test_merge_subnormal_accumulator(orc):
    """B A and W' in the fp32 subnormal range: the merge must not flush them."""
    require_gpu()
    g = torch.Generator().manual_seed(23)
    N, K = 96, 192
    W = torch.randn(N, K, generator=g) * 1e-39
    A = torch.randn(32, K, generator=g) * 1e-20
    B = torch.randn(N, 32, generator=g) * 1e-19
    _check_merge(orc, W, A, B, 32.0)
    _check_merge(orc, W * 0, A, B, 0.5)
    _check_requant(orc, W, A, B, 32.0)


def test_requant_back_to_back_calls_are_stable(orc):
    """Forty back-to-back requants of the FLUX.1-shaped weight on one stream (each one
    kernel with a grid-wide barrier between its amax and quantize phases), every
    result bit-identical to the oracle's: a barrier that let a CTA read the amax early,
    or a stale tile, would show up as a mismatch in some call."""
    require_gpu()
    cfg = workloads.LINEARS["flux_up"]
    W = workloads.weight(cfg, seed=3)
    A, B = workloads.lora(cfg, seed=3)
    Wd, Ad, Bd = W.cuda(), A.cuda(), B.cuda()
    N, K = cfg.N, cfg.K
    outs = [(torch.empty(N, K // 2, dtype=torch.uint8, device="cuda"),
             torch.empty(nv.sf_bytes(N, K), dtype=torch.uint8, device="cuda"),
             torch.empty(1, dtype=torch.float32, device="cuda")) for _ in range(40)]
    ws = torch.empty(nv.requant_workspace_bytes(nv.W_BF16, 32, N, K), dtype=torch.uint8, device="cuda")
    for o in outs:
        nv.nvfp4_requant(Wd, Ad, Bd, workloads.LORA_ALPHA, *o, workspace=ws)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_status() == 0
    oc, osf, os_ = orc.requant(workloads.bf16_bits(W), A.numpy(), B.numpy(), workloads.LORA_ALPHA)
    first = [np_(t) for t in outs[0]]
    sf_rm, _ = unswizzle_sf(first[1], N, K)
    assert first[2].view(np.uint32)[0] == os_.view(np.uint32)[0]
    assert np.array_equal(sf_rm, osf) and np.array_equal(first[0], oc)
    for j, o in enumerate(outs[1:], 1):
        for a, b in zip(first, (np_(t) for t in o)):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"call {j} differs from call 0"
