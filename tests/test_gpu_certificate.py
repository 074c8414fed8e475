"""Adversarial parity for the tensor-core requant's certified decisions.

The tensor-core path of nvfp4_requant computes the LoRA term B A with bf16-split
products on the tensor cores and takes each decision (the tensor amax, a block's
E4M3 scale, an element's E2M1 code) only where an error bound certifies it; every
other decision is recomputed with the exact fp32 chain.  Random weights put few
merged values near a decision, so here W, A and B are built so that a large share
of the merged values w' (NVIDIA NVFP4 blog, "two-level scaling"; Sol-RL project
page, "Two-Stage Pipeline", Stage 2: merge, then re-quantize) land within a few
fp32 ulps of a decision boundary:

  * the per-tensor scale is pinned: one element, with no LoRA term (its column of A
    is zero), is 2688 * 2^-12, the largest |w'|, so s = 2^-12 exactly;
  * "code" rows: every 16-element block holds, in its first column (no LoRA term),
    6 v s for an E4M3 value v, so the block scale is exactly v; the other 15
    elements are W = m v s for an E2M1 rounding midpoint m in {0.25, 0.75, 1.25,
    1.75, 2.5, 3.5, 5}, i.e. on a code boundary times den = v s, and the LoRA term
    moves them by a few ulps (sometimes by less than half an ulp: an exact tie);
  * "scale" rows: each block's largest element is 6 mu s for mu the midpoint of two
    neighbouring E4M3 values, so the LoRA term decides the block scale by a few ulps.

The LoRA term's size is set per row and column (powers of two times N(0, 1)
factors) so that |c (B A)[n, k]| spans about 2^-3 .. 2^10 ulps of W[n, k].  A
second family plants near-maximal competitors in realistic weights, so that the
tensor amax itself is decided among values a few ulps apart.

Every output must be bit-identical to the oracle's.  Each case also reports how
many elements the kernel sent to the exact chain (nvfp4_requant_exact_counts).
E4M3 and E2M1 values below are written from the OCP MX format definitions.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import np_, require_gpu, unswizzle_sf

pytestmark = pytest.mark.gpu

R = 32
S_EXP = -12
E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _e4m3_values():
    """Positive finite E4M3 values in increasing order: subnormals m/8 * 2^-6, then
    (1 + m/8) 2^(e-7) for e = 1..15, the top code (e = 15, m = 7) being NaN."""
    vals = [m / 8 * 2.0 ** -6 for m in range(1, 8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


E4M3 = _e4m3_values()
assert E4M3[-1] == 448.0


def _bf16(x64):
    """float64 values that are exactly representable in bf16 -> torch bf16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(x64, np.float32))
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "construction produced a value that is not a bf16"
    return b


def build_boundary_case(N, K, seed):
    """(W bf16 [N, K], A fp32 [R, K], B fp32 [N, R]) as described in the module doc."""
    rng = np.random.default_rng(seed)
    s = 2.0 ** S_EXP
    c = workloads.LORA_ALPHA / R
    W = np.zeros((N, K))
    nblk = K // 16
    scale_row = rng.random(N) < 0.3
    scale_row[0] = False
    # Block scales: mostly normal E4M3 values from 2^-3 up to 448, a few subnormals.
    idx_lo, idx_hi = int(np.searchsorted(E4M3, 2.0 ** -3)), len(E4M3) - 2
    vi = rng.integers(idx_lo, idx_hi + 1, N)
    sub = rng.random(N) < 0.05
    vi[sub] = rng.integers(0, 7, int(sub.sum()))
    vi[0] = len(E4M3) - 1                                   # row 0: v = 448, the amax anchor
    v = E4M3[vi]
    sign = rng.choice([-1.0, 1.0], (N, K))
    m = E2M1_MIDPOINTS[rng.integers(0, len(E2M1_MIDPOINTS), (N, K))]
    for n in range(N):
        if not scale_row[n]:
            W[n] = sign[n] * m[n] * v[n] * s
            W[n, ::16] = 6.0 * v[n] * s                     # the block's scale anchor
        else:
            mu = 0.5 * (v[n] + E4M3[vi[n] + 1])
            mm = np.minimum(m[n], 3.5)
            W[n] = sign[n] * mm * v[n] * s
            W[n, ::16] = 0.0
            pos = rng.integers(1, 16, nblk) + 16 * np.arange(nblk)
            W[n, pos] = sign[n, pos] * 6.0 * mu * s         # the block's largest, on a scale midpoint
    Wb = _bf16(W)
    # LoRA factors: column k's A scaled by 2^omega_k (zero on the anchor columns), row
    # n's B by 2^tau_n times the ulp of the row's typical |W|.
    omega = rng.uniform(-2.0, 2.0, K)
    a_scale = 2.0 ** omega
    a_scale[::16] = 0.0
    A = rng.standard_normal((R, K)) * a_scale[None, :]
    row_ref = np.where(scale_row, 6.0 * v, 1.25 * v) * s
    ulp_row = 2.0 ** (np.floor(np.log2(row_ref)) - 23)
    tau = rng.uniform(-3.0, 10.0, N)
    b_scale = ulp_row * 2.0 ** tau / (c * np.sqrt(R))
    B = rng.standard_normal((N, R)) * b_scale[:, None]
    return Wb, torch.from_numpy(A.astype(np.float32)), torch.from_numpy(B.astype(np.float32))


def build_amax_case(N, K, seed):
    """Realistic weights with 64 planted competitors for the tensor amax: the same
    bf16 value (above every other |W|), each moved by its own LoRA term by a few ulps
    up or down, so that the maximum is decided among values a few ulps apart."""
    cfg = workloads.LinearConfig(name="amax_case", M=128, K=K, N=N)
    W = workloads.weight(cfg, seed=seed).float().numpy().astype(np.float64)
    rng = np.random.default_rng(seed + 1000)
    top = float(np.abs(W).max())
    peak = float(_bf16(np.array([2.0 ** np.ceil(np.log2(top * 1.5))])).float()[0])
    flat = rng.choice(N * K, 64, replace=False)
    W.reshape(-1)[flat] = peak * rng.choice([-1.0, 1.0], 64)
    Wb = _bf16(W)
    c = workloads.LORA_ALPHA / R
    ulp = 2.0 ** (np.floor(np.log2(peak)) - 23)
    A = rng.standard_normal((R, K)) * 2.0 ** rng.uniform(-1.0, 1.0, K)[None, :]
    B = rng.standard_normal((N, R)) * (ulp * 2.0 ** rng.uniform(-2.0, 4.0, N) / (c * np.sqrt(R)))[:, None]
    return Wb, torch.from_numpy(A.astype(np.float32)), torch.from_numpy(B.astype(np.float32))


def build_amax_flood_case(N, K, seed):
    """Every |W| within 3 bf16 steps of the top (0.5 - j 2^-9, j = 0..3) and a LoRA
    term whose bound spans about two of those steps: most elements stay candidates for
    the tensor amax to the end, so every CTA's candidate queue overflows and the amax
    phase finishes in its slow mode (candidates merged where they are found)."""
    rng = np.random.default_rng(seed)
    j = rng.integers(0, 4, (N, K))
    W = (0.5 - j * 2.0 ** -9) * rng.choice([-1.0, 1.0], (N, K))
    A = rng.standard_normal((R, K)) / 32
    B = rng.standard_normal((N, R)) * (2.0 ** -8 / 1.4)
    c = workloads.LORA_ALPHA / R
    B /= c
    return _bf16(W), torch.from_numpy(A.astype(np.float32)), torch.from_numpy(B.astype(np.float32))


def _ulps(x, target):
    """|x - target| in fp32 ulps of x (x float32, target float64)."""
    return np.abs(x.astype(np.float64) - target) / np.spacing(np.abs(x)).astype(np.float64)


def near_boundary_counts(wp, sf, s_t):
    """From the oracle's merged values and its outputs: how many elements lie within
    1-16 ulps (and within less than 1 ulp) of an E2M1 boundary times den, and how many
    blocks have their largest |w'| within 1-16 ulps of an E4M3 midpoint times 6 s."""
    N, K = wp.shape
    s = float(s_t[0])
    sfv = np.concatenate([[0.0], E4M3])
    den = np.repeat(_e4m3_decode(sf), 16, axis=1) * s
    live = den > 0
    q = np.abs(wp.astype(np.float64)) / np.where(live, den, 1.0)
    j = np.clip(np.searchsorted(E2M1_MIDPOINTS, q), 1, len(E2M1_MIDPOINTS) - 1)
    lo, hi = E2M1_MIDPOINTS[j - 1], E2M1_MIDPOINTS[j]
    mid = np.where(np.abs(q - lo) <= np.abs(q - hi), lo, hi)
    d = np.where(live & (wp != 0), _ulps(np.abs(wp), mid * den), np.inf)
    code_near = int(((d >= 1) & (d <= 16)).sum())
    code_sub = int((d < 1).sum())
    bam = np.abs(wp).reshape(N, K // 16, 16).max(axis=2)
    mids = 0.5 * (sfv[:-1] + sfv[1:]) * 6.0 * s
    j = np.clip(np.searchsorted(mids, bam.astype(np.float64)), 1, len(mids) - 1)
    dist = np.minimum(_ulps(bam, mids[j - 1]), _ulps(bam, mids[j]))
    dist = np.where(bam > 0, dist, np.inf)
    scale_near = int(((dist >= 1) & (dist <= 16)).sum() + (dist < 1).sum())
    return code_near, code_sub, scale_near


def _e4m3_decode(codes):
    codes = np.asarray(codes, np.int64)
    e, m = (codes >> 3) & 0xF, codes & 7
    val = np.where(e == 0, m / 8 * 2.0 ** -6, (1 + m / 8) * 2.0 ** (e - 7))
    return np.where(codes & 0x80, -val, val)


def _run(orc, W, A, B):
    N, K = W.shape
    ws = torch.empty(nv.requant_workspace_bytes(nv.W_BF16, R, N, K), dtype=torch.uint8, device="cuda")
    codes, sf, s_t = nv.nvfp4_requant(W.cuda(), A.cuda(), B.cuda(), workloads.LORA_ALPHA, workspace=ws)
    torch.cuda.synchronize()
    counts = nv.nvfp4_requant_exact_counts(ws, N, K)
    codes, sf, s_t = np_(codes), np_(sf), np_(s_t)
    sf_rm, sf_pad = unswizzle_sf(sf, N, K)
    Wn = workloads.bf16_bits(W)
    oc, osf, os_ = orc.requant(Wn, A.numpy(), B.numpy(), workloads.LORA_ALPHA)
    assert s_t.view(np.uint32)[0] == os_.view(np.uint32)[0], f"s_t {s_t[0]!r} vs {os_[0]!r}"
    assert not sf_pad.any(), "scale padding rows must be zero"
    assert np.array_equal(sf_rm, osf), f"block scales differ at {np.argwhere(sf_rm != osf)[:3]}"
    assert np.array_equal(codes, oc), f"codes differ at {np.argwhere(codes != oc)[:3]}"
    assert nv.nvfp4_device_status() == 0
    wp = orc.merge(Wn, A.numpy(), B.numpy(), workloads.LORA_ALPHA)
    return counts, wp, osf, os_


@pytest.mark.parametrize("N,K", [(256, 12288), (520, 3072), (384, 2240)])
@pytest.mark.parametrize("seed", range(20))
def test_certificate_on_boundaries(orc, N, K, seed):
    require_gpu()
    if (N, K) != (256, 12288) and seed >= 8:
        pytest.skip("8 seeds for the smaller shapes")
    W, A, B = build_boundary_case(N, K, seed)
    (xq, xa), wp, osf, os_ = _run(orc, W, A, B)
    assert os_[0] == np.float32(2.0 ** S_EXP), "the amax anchor must fix s"
    code_near, code_sub, scale_near = near_boundary_counts(wp, osf, os_)
    print(f"\n[certificate N={N} K={K} seed={seed}] elements within 1-16 ulps of a code boundary: "
          f"{code_near}, within <1 ulp: {code_sub}; blocks within 16 ulps of a scale midpoint: "
          f"{scale_near}; exact chain: {xq} quantize-phase elements, {xa} amax candidates")
    # The construction does what it claims (thousands of elements per case).
    assert code_near >= N * K // 64, code_near
    assert scale_near >= N * K // 16 // 64, scale_near
    assert xq > 0, "the exact fallback must have been exercised"


@pytest.mark.parametrize("seed", range(20))
def test_certificate_amax_competitors(orc, seed):
    require_gpu()
    N, K = (256, 3072) if seed % 2 == 0 else (264, 12288)
    W, A, B = build_amax_case(N, K, seed)
    (xq, xa), wp, osf, os_ = _run(orc, W, A, B)
    top = np.sort(np.abs(wp).reshape(-1))[-64:]
    spread = _ulps(top[-1:], top[0].astype(np.float64))[0]
    print(f"\n[amax N={N} K={K} seed={seed}] 64 competitors span {spread:.0f} ulps; "
          f"exact chain: {xa} amax candidates, {xq} quantize-phase elements")
    assert spread <= 1024, spread
    assert xa > 0, "the amax candidates must have been merged exactly"


@pytest.mark.parametrize("N,K,seed", [(1024, 3072, 0), (520, 2240, 1), (256, 12288, 2)])
def test_certificate_amax_queue_overflow(orc, N, K, seed):
    """The amax phase's slow mode: thousands of candidates per CTA."""
    require_gpu()
    W, A, B = build_amax_flood_case(N, K, seed)
    (xq, xa), wp, osf, os_ = _run(orc, W, A, B)
    print(f"\n[amax flood N={N} K={K} seed={seed}] exact chain: {xa} amax candidates, {xq} quantize-phase elements")
    assert xa > 512 * 4, "the candidate queues must have overflowed"
